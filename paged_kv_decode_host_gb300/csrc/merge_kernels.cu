// Attention-state merge kernels for sm_103a.
//
// The algebra (FlashInfer 完全拆解, 在线 Softmax 为什么允许任意切块; FlashInfer,
// in depth, "Load balancing with split-KV"): states (O_I, L_I) over disjoint
// key sets combine exactly as M = max L, w = exp(L - M), O = sum w O / sum w,
// L = M + log sum w.  Both kernels are HBM/latency-bound elementwise passes;
// neither uses atomics, and each output is produced by one fixed sequence of
// floating-point operations, so results are bit-reproducible.
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "pkd_internal.h"

namespace pkd {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994530942f;

__device__ __forceinline__ uint32_t f32_to_bf16_rne(float x) {
  uint32_t u = __float_as_uint(x);
  if ((u & 0x7fffffffu) > 0x7f800000u) return 0x7fc0u;
  u += 0x7fffu + ((u >> 16) & 1u);
  return u >> 16;
}

__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Contraction of split chunks (the reduction map built by the planner): for
// each split request u and query head h, fold the partial states in slots
// merge_indptr[u] .. merge_indptr[u+1] into out / lse.  Block = 256 threads
// = 8 warps, grid = 8 blocks per decode CTA; (unit, head) tasks:
//  * one block per task by default: the block first takes M = max L over the
//    unit's chunks, then warp w sums exp(L - M) O and exp(L - M) over slots
//    w, w + 8, ... (lane = 4 dims); the 8 warp sums are added in warp order;
//  * with at least 4 tasks per block (hundreds of split requests), one warp
//    per task for units of at most 32 chunks: lane i reads chunk i's L, the
//    warp takes M and the weights w_i = exp(L_i - M) with shuffles, then
//    every lane sums w_i O_i over its 4 dims -- no block barrier; longer
//    units still get a block.  (Measured: with few tasks the block form is
//    the faster one, as every block then carries work.)
// With M known up front no term rescales a running sum, so the loads of a
// warp can stay in flight together.  kBatch > 1 (plans that split a request
// into more than kLongUnit chunks) makes that explicit in the block path: a
// warp issues the loads of kBatch slots before adding their terms (the first
// batch's already before the max pass), so a 250-chunk request costs a few
// memory round trips per warp instead of one per slot; it needs more registers (fewer resident blocks), which plans of
// short units do not repay, so they get kBatch = 1.  The terms are added in
// the same order either way.  Fixed assignment and order: bit-reproducible.
// Cascade plans (every request one unit of its prefix and suffix chunks, at
// most 32) take kBatch = 4; with at most 16 chunks in 4-warp blocks, so
// that the grid's blocks (64 registers a thread at 8 warps would allow four
// per SM, two waves for the shared-prefix step's 1,024 tasks) are all
// resident at once.
constexpr int kWarpSlots = 32;

template <int kBatch, int kThreads = kMergeThreads>
__global__ void __launch_bounds__(kThreads) merge_partials_kernel(const MergeArgs a) {
  static_assert(kThreads >= kHeadDim && kThreads % 32 == 0, "a thread per output dim");
  constexpr int kWarps = kThreads / 32;
  __shared__ float wm[kWarps];
  __shared__ float wz[kWarps];
  __shared__ __align__(16) float wacc[kWarps][kHeadDim];
  pdl_launch_dependents();
  // The schedule is written by host-to-device copies.  When the stream
  // orders them before this kernel, read it before waiting for the decode
  // kernel; when the plan came from another stream (wait_epoch), the decode
  // kernel waited for it, so read it once that grid has completed.
  bool waited = false;
  if (a.wait_epoch != 0) {
    pdl_wait();
    waited = true;
  }
  const int n_units = a.sched[H_NUNITS];
  const int64_t tasks = (int64_t)n_units * a.hq;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool warp_mode = tasks >= (int64_t)4 * gridDim.x;
  // ---- short units, many tasks: a warp per task
  const int64_t n_warps = (int64_t)gridDim.x * kWarps;
  const int64_t warp_tasks = warp_mode ? tasks : 0;
  for (int64_t task = (int64_t)blockIdx.x * kWarps + warp; task < warp_tasks; task += n_warps) {
    const int u = (int)(task / a.hq);
    const int h = (int)(task % a.hq);
    const int s0 = a.sched[a.off_merge + u];
    const int n = a.sched[a.off_merge + u + 1] - s0;
    if (n > kWarpSlots) continue;
    const int req = a.sched[a.off_units + 2 * u];
    if (!waited) {
      pdl_wait();   // partial states and outputs belong to the decode kernel
      waited = true;
    }
    const float l2 = lane < n ? a.l_part[(int64_t)(s0 + lane) * a.hq + h] * kLog2e : -CUDART_INF_F;
    float m = l2;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float w_lane = lane < n ? exp2f(l2 - m) : 0.f;
    float z = w_lane;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
    for (int i = 0; i < n; ++i) {
      const float w = __shfl_sync(0xffffffffu, w_lane, i);
      const float4 o = *reinterpret_cast<const float4*>(
          a.o_part + ((int64_t)(s0 + i) * a.hq + h) * kHeadDim + 4 * lane);
      acc.x = fmaf(w, o.x, acc.x);
      acc.y = fmaf(w, o.y, acc.y);
      acc.z = fmaf(w, o.z, acc.z);
      acc.w = fmaf(w, o.w, acc.w);
    }
    const float inv = 1.f / z;
    const int64_t qrow = (int64_t)req * a.hq + h;
    *reinterpret_cast<uint2*>(a.out + qrow * kHeadDim + 4 * lane) =
        make_uint2(f32_to_bf16_rne(acc.x * inv) | (f32_to_bf16_rne(acc.y * inv) << 16),
                   f32_to_bf16_rne(acc.z * inv) | (f32_to_bf16_rne(acc.w * inv) << 16));
    if (lane == 0 && a.lse != nullptr) a.lse[qrow] = (m + log2f(z)) * kLn2;
  }
  // ---- a block per task (in warp mode only the long units, and only when
  // the plan has any)
  const int64_t block_tasks =
      (!warp_mode || a.sched[H_MAXCHUNKS] > kWarpSlots) ? tasks : 0;
  for (int64_t task = blockIdx.x; task < block_tasks; task += gridDim.x) {
    const int u = (int)(task / a.hq);
    const int h = (int)(task % a.hq);
    const int s0 = a.sched[a.off_merge + u];
    const int s1 = a.sched[a.off_merge + u + 1];
    if (warp_mode && s1 - s0 <= kWarpSlots) continue;   // the same for the whole block
    const int req = a.sched[a.off_units + 2 * u];
    if (!waited) {
      pdl_wait();
      waited = true;
    }
    // kBatch > 1: this warp's first batch of slots is loaded before pass 1,
    // so its round trip overlaps the max pass's
    float lv[kBatch];
    float4 ov[kBatch];
    auto load_batch = [&](int base) {
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int s = base + j * kWarps;
        if (s < s1) {
          lv[j] = a.l_part[(int64_t)s * a.hq + h];
          ov[j] = *reinterpret_cast<const float4*>(a.o_part + ((int64_t)s * a.hq + h) * kHeadDim +
                                                   4 * lane);
        } else {
          lv[j] = -CUDART_INF_F;   // weight 0
          ov[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
    };
    if constexpr (kBatch > 1) load_batch(s0 + warp);
    // ---- pass 1: M = max over the unit's chunk LSEs (log2 units)
    float mx = -CUDART_INF_F;
    for (int s = s0 + threadIdx.x; s < s1; s += kThreads)
      mx = fmaxf(mx, a.l_part[(int64_t)s * a.hq + h] * kLog2e);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) wm[warp] = mx;
    __syncthreads();
    float m = wm[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w) m = fmaxf(m, wm[w]);
    // ---- pass 2: this warp's share of sum exp2(L - M) O and sum exp2(L - M)
    // slots w, w + kWarps, ... (in batches of kBatch: a batch's loads are all
    // issued before its terms are added, in the same order)
    float z = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if constexpr (kBatch == 1) {
#pragma unroll 8
      for (int s = s0 + warp; s < s1; s += kWarps) {
        const float w = exp2f(a.l_part[(int64_t)s * a.hq + h] * kLog2e - m);
        const float4 o = *reinterpret_cast<const float4*>(
            a.o_part + ((int64_t)s * a.hq + h) * kHeadDim + 4 * lane);
        acc.x = fmaf(w, o.x, acc.x);
        acc.y = fmaf(w, o.y, acc.y);
        acc.z = fmaf(w, o.z, acc.z);
        acc.w = fmaf(w, o.w, acc.w);
        z += w;
      }
    }
    for (int base = s0 + warp; kBatch > 1 && base < s1; base += kBatch * kWarps) {
      if (base != s0 + warp) load_batch(base);
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const float w = exp2f(lv[j] * kLog2e - m);
        acc.x = fmaf(w, ov[j].x, acc.x);
        acc.y = fmaf(w, ov[j].y, acc.y);
        acc.z = fmaf(w, ov[j].z, acc.z);
        acc.w = fmaf(w, ov[j].w, acc.w);
        z += w;
      }
    }
    *reinterpret_cast<float4*>(&wacc[warp][4 * lane]) = acc;
    if (lane == 0) wz[warp] = z;
    __syncthreads();
    if (threadIdx.x < kHeadDim) {
      float o = 0.f, zt = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        o += wacc[w][threadIdx.x];
        zt += wz[w];
      }
      const int64_t qrow = (int64_t)req * a.hq + h;
      a.out[qrow * kHeadDim + threadIdx.x] = (uint16_t)f32_to_bf16_rne(o / zt);
      if (threadIdx.x == 0 && a.lse != nullptr) a.lse[qrow] = (m + log2f(zt)) * kLn2;
    }
    __syncthreads();
  }
  if (!waited) pdl_wait();
}

// merge_states: two states per row, row = (n, head), rows_per_block rows of
// head_dim / 8 threads each (one 16-byte chunk of 8 bf16 per thread).
__global__ void __launch_bounds__(256) merge_states_kernel(
    const uint16_t* __restrict__ va, const float* sa, const uint16_t* __restrict__ vb,
    const float* sb, uint16_t* vo, float* so, int64_t rows, int chunks, int rows_per_block) {
  const int r_local = threadIdx.x / chunks;
  const int c = threadIdx.x % chunks;
  const int64_t r = (int64_t)blockIdx.x * rows_per_block + r_local;
  const bool active = r_local < rows_per_block && r < rows;
  float la = 0.f, lb = 0.f;
  uint4 xa = make_uint4(0, 0, 0, 0), xb = xa;
  if (active) {
    la = sa[r];
    lb = sb[r];
    xa = *reinterpret_cast<const uint4*>(va + (r * chunks + c) * 8);
    xb = *reinterpret_cast<const uint4*>(vb + (r * chunks + c) * 8);
  }
  __syncthreads();  // every read of s_a / s_b / v happens before any write (aliasing)
  if (!active) return;
  const float m = fmaxf(la, lb);
  uint4 res = make_uint4(0, 0, 0, 0);
  float lse = -CUDART_INF_F;
  if (m != -CUDART_INF_F) {
    const float wa = exp2f((la - m) * kLog2e);
    const float wb = exp2f((lb - m) * kLog2e);
    const float z = wa + wb;
    const float inv = 1.f / z;
    const uint32_t a4[4] = {xa.x, xa.y, xa.z, xa.w};
    const uint32_t b4[4] = {xb.x, xb.y, xb.z, xb.w};
    uint32_t o4[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float a0 = __uint_as_float(a4[k] << 16), a1 = __uint_as_float(a4[k] & 0xffff0000u);
      const float b0 = __uint_as_float(b4[k] << 16), b1 = __uint_as_float(b4[k] & 0xffff0000u);
      const float o0 = (wa * a0 + wb * b0) * inv;
      const float o1 = (wa * a1 + wb * b1) * inv;
      o4[k] = f32_to_bf16_rne(o0) | (f32_to_bf16_rne(o1) << 16);
    }
    res = make_uint4(o4[0], o4[1], o4[2], o4[3]);
    lse = m + log2f(z) * kLn2;
  }
  *reinterpret_cast<uint4*>(vo + (r * chunks + c) * 8) = res;
  if (c == 0) so[r] = lse;
}

}  // namespace

cudaError_t launch_merge_partials(const MergeArgs& a, int grid, int32_t max_chunks,
                                  cudaStream_t stream, bool batch_short) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kMergeThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (max_chunks > kLongUnit) return cudaLaunchKernelEx(&cfg, merge_partials_kernel<8>, a);
  if (batch_short && max_chunks <= 4 * 4) {
    // 4-warp blocks: at 64 registers a thread, eight of them fit an SM, so
    // the grid's blocks are all resident at once
    cfg.blockDim = dim3(128);
    return cudaLaunchKernelEx(&cfg, merge_partials_kernel<4, 128>, a);
  }
  if (batch_short && max_chunks <= 4 * (kMergeThreads / 32))
    return cudaLaunchKernelEx(&cfg, merge_partials_kernel<4>, a);
  return cudaLaunchKernelEx(&cfg, merge_partials_kernel<1>, a);
}

cudaError_t launch_merge_states(const void* v_a, const float* s_a, const void* v_b,
                                const float* s_b, void* v_out, float* s_out, int64_t rows,
                                int head_dim, cudaStream_t stream) {
  const int chunks = head_dim / 8;
  const int rows_per_block = 256 / chunks;
  const int64_t blocks = (rows + rows_per_block - 1) / rows_per_block;
  merge_states_kernel<<<(unsigned)blocks, 256, 0, stream>>>(
      static_cast<const uint16_t*>(v_a), s_a, static_cast<const uint16_t*>(v_b), s_b,
      static_cast<uint16_t*>(v_out), s_out, rows, chunks, rows_per_block);
  return cudaGetLastError();
}

}  // namespace pkd
