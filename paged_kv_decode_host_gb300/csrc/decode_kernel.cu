// Persistent paged-KV decode kernel for sm_103a.
//
// What it computes (FlashInfer 完全拆解, 从推理形状出发 and 在线 Softmax 为什么
// 允许任意切块; FlashInfer, in depth, "GQA, tensor cores and MLA"): for each
// work item (request, page-aligned token range) of this CTA's queue, the
// attention state of every query head of the request over those tokens,
//   s_t = q . k_t / sqrt(D),  O = sum_t exp(s_t - m) v_t / sum_t exp(s_t - m),
//   L = m + log sum_t exp(s_t - m),
// streamed with the online-softmax recurrence so scores never reach HBM.
// Unsplit items write (O, L) straight to out / lse ("writethrough"); chunks
// of split requests write (O, L) to their partial slot for the merge kernel.
//
// GB300 design:
//  * Grid = the plan's fixed CTA count (persistent; only the queue contents
//    change between plans, so launches can be captured in a CUDA graph).
//  * One producer warp streams the item's tokens into a ring of shared-memory
//    stages with TMA (completion on an mbarrier, L2 evict-first): two stages
//    deep for the bf16 tensor-core consumer, three for the others
//    (ring_depth).  A stage holds 16 tokens (32 for an e4m3 cache).  Two
//    producers:
//      - page tiles (page size a multiple of 16): one tensor-map copy
//        (cp.async.bulk.tensor, 5-D) moves 16 tokens of K (or V) of all KV
//        heads, re-ordered to [head][128-byte half][token] with the 128-byte
//        swizzle, so 8-token fragment loads of one head are conflict-free;
//      - token rows (any page size): in the NHD layout one token row of all
//        KV heads is contiguous, so each token costs one K-row and one V-row
//        bulk copy (cp.async.bulk, 2 KiB each at 8 KV heads), landing at a
//        padded row stride for the same reason (HND: one copy per token and
//        KV head).  Only valid rows are copied.
//    Both producers read either cache layout (NHD [pages][2][P][Hkv][D] or
//    HND [pages][2][Hkv][P][D]) into the same shared-memory layout, so the
//    consumers do not depend on it.
//  * One consumer warp per KV head folds its GQA group of G query heads onto
//    each K/V row it reads from shared memory (one read serves G heads).  The
//    default consumer runs the group as a thin matrix on tensor cores
//    (mma.sync m16n8k16, bf16 in, fp32 accumulate); the CUDA-core consumer
//    (fp32 FMA, lanes split D, reduce-scatter of the dot products across a
//    half-warp) is kept as an option.  Softmax statistics are fp32.
//  * Programmatic dependent launch: CTAs trigger the next kernel at start; the
//    producer streams KV tiles at once, the tensor-core consumers read q at
//    once and wait for the previous kernel only before their first write of
//    outputs or partial states (see the note in decode_kernel).
//  * Every wait is bounded (~2 s of %globaltimer); on timeout the kernel sets
//    the device error word, stops issuing copies, waits (bounded) for the
//    copies already in flight, and returns.
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <cuda_fp8.h>
#include <math_constants.h>
#include <stdint.h>

#include <mutex>

#include "pkd_internal.h"
#include "prefix_tc_body.cuh"
#include "sm103_ptx.cuh"

namespace pkd {
namespace {

using namespace dev;

constexpr int kTS = kWarpTokens;                 // tokens per stage
// Shared-memory stride of one token row (all KV heads): 16 bytes of padding
// shift consecutive rows across banks, so 8-row fragment loads of one head
// are conflict-free.
__host__ __device__ __forceinline__ int row_stride(int row_bytes) { return row_bytes + 16; }

// Token-row stage geometry: token t's K row at t * tok_stride and its V row
// at v_base + t * tok_stride.  Separate copies: all K rows, then all V rows,
// each at the padded row stride.  Merged copies (page size 1, where a
// token's K and V rows are adjacent in the cache): [K row | V row] per token
// at stride 2 row + 16, so one copy moves both.  Both strides are 16 bytes
// past a multiple of 128: 8-row fragment loads stay conflict-free.
__device__ __forceinline__ int rows_tok_stride(const DecodeArgs& a) {
  return a.kv_merged ? 2 * a.row_bytes + 16 : row_stride(a.row_bytes);
}
__device__ __forceinline__ int rows_v_base(const DecodeArgs& a, int tokens) {
  return a.kv_merged ? a.row_bytes : tokens * row_stride(a.row_bytes);
}

// 8 bf16 (one uint4) -> 8 fp32, exact.
__device__ __forceinline__ void bf16x8_to_f32(const uint4 r, float (&f)[8]) {
  const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// fp32 -> bf16 bits, round to nearest even (finite inputs; NaN kept NaN).
__device__ __forceinline__ uint32_t f32_to_bf16_rne(float x) {
  uint32_t u = __float_as_uint(x);
  if ((u & 0x7fffffffu) > 0x7f800000u) return 0x7fc0u;
  u += 0x7fffu + ((u >> 16) & 1u);
  return u >> 16;
}

// One reduce-scatter level across lanes `mask` apart: lanes with the mask
// bit set keep the upper half of v, the others the lower half; each adds the
// partner's copy of the half it keeps.
template <int N>
__device__ __forceinline__ void rs_level(const float (&v)[N], float (&o)[N / 2], int mask,
                                         bool upper) {
#pragma unroll
  for (int t = 0; t < N / 2; ++t) {
    const float keep = upper ? v[N / 2 + t] : v[t];
    const float send = upper ? v[t] : v[N / 2 + t];
    o[t] = keep + __shfl_xor_sync(kFull, send, mask);
  }
}

// ---------------------------------------------------------------- producer
// Page tiles (kTiles): stage = [K box 0 .. kBoxes-1][V box 0 .. kBoxes-1],
// box b holding tokens 16 b .. 16 b + 15 of the stage as [head][half][token]
// lines of 128 bytes; lane 2 b + c copies box b of K (c = 0) or V (c = 1).
// A box always moves 16 token slots of its page; slots past the item's end
// are in-page bytes the consumers mask (scores) or zero (V).
// Token rows: stage = [K rows][V rows] at the padded row stride; lane j
// copies token j's K row and V row (valid tokens only).
template <int kTokens, bool kTiles, int kRing>
__device__ void run_producer(const DecodeArgs& a, int it0, int it1, uint8_t* stages,
                             int stage_bytes, uint64_t* full, uint64_t* empty,
                             volatile int* abort_flag, int lane) {
  constexpr int kBoxes = kTokens / 16;
  const int P = a.page_size;
  const int row = a.row_bytes;
  const int rs = rows_tok_stride(a);
  const int vb = rows_v_base(a, kTokens);
  const uint32_t box = (uint32_t)(16 * row);
  const uint64_t policy = l2_evict_first_policy();
  uint32_t stage = 0;
  bool ok = true;
  for (int it = it0; it < it1 && ok; ++it) {
    const int32_t* item = a.sched + a.off_items + (int64_t)it * kItemWords;
    const int tb = item[1], te = item[2], poff = item[4];
    for (int t = tb; t < te; t += kTokens) {
      const int n = min(kTokens, te - t);
      const int slot = (int)(stage % kRing);
      const uint32_t round = stage / kRing;
      // this lane's token (rows) or box (tiles), and its page id
      const int nbox = (n + 15) >> 4;
      const int tok = kTiles ? t + 16 * (lane >> 1) : t + lane;
      int page = -1;
      if (kTiles ? (lane >> 1) < nbox : lane < n) {
        page = a.sched[a.off_pages + poff + (tok - tb) / P];
        if ((unsigned)page >= (unsigned)a.num_pages) {
          atomicOr(a.err, PKD_DEV_ERR_BOUNDS);
          page = 0;
        }
      }
      if (round > 0) {
        bool w = mbar_wait(&empty[slot], (round - 1) & 1u, abort_flag);
        if (!__all_sync(kFull, w)) {
          if (lane == 0) raise_error(a.err, abort_flag, PKD_DEV_ERR_TIMEOUT);
          ok = false;
          break;
        }
      }
      if (lane == 0)
        mbar_arrive_expect_tx(&full[slot], kTiles ? 2u * (uint32_t)nbox * box
                                                  : (uint32_t)(2 * n * row));
      __syncwarp();
      if (page >= 0) {
        uint8_t* st = stages + (size_t)slot * stage_bytes;
        if constexpr (kTiles) {
          const int c = lane & 1;
          tensor_copy_g2s(st + (size_t)(c * kBoxes + (lane >> 1)) * box, &a.kv_map, 0, tok % P, 0,
                          0, 2 * page + c, &full[slot], policy);
        } else {
          uint8_t* dk = st + (size_t)lane * rs;
          uint8_t* dv = st + vb + (size_t)lane * rs;
          if (a.kv_merged) {
            // page size 1: K row and V row back to back, one copy
            bulk_copy_g2s(dk, a.kv + (int64_t)page * a.page_bytes, (uint32_t)(2 * row), &full[slot],
                          policy);
          } else if (!a.hnd) {
            const uint8_t* src = a.kv + (int64_t)page * a.page_bytes + (int64_t)(tok % P) * row;
            bulk_copy_g2s(dk, src, (uint32_t)row, &full[slot], policy);
            bulk_copy_g2s(dv, src + (int64_t)P * row, (uint32_t)row, &full[slot], policy);
          } else {
            // HND: the token's KV heads sit P rows of one head apart
            const int hb = row / a.hkv;
            const uint8_t* src = a.kv + (int64_t)page * a.page_bytes + (int64_t)(tok % P) * hb;
            for (int h = 0; h < a.hkv; ++h) {
              const uint8_t* sk = src + (int64_t)h * P * hb;
              bulk_copy_g2s(dk + h * hb, sk, (uint32_t)hb, &full[slot], policy);
              bulk_copy_g2s(dv + h * hb, sk + (int64_t)P * row, (uint32_t)hb, &full[slot],
                            policy);
            }
          }
        }
      }
      ++stage;
    }
  }
  pdl_wait();   // complete only after the previous kernel (see the kernel's note)
  // Drain: wait for the last issued phase of every slot, so no copy is in
  // flight into shared memory when the CTA exits.
  if (lane == 0) {
    for (uint32_t s = 0; s < (uint32_t)kRing; ++s) {
      if (stage > s) {
        const uint32_t last_round = (stage - 1 - s) / kRing;
        if (!mbar_wait(&full[s], last_round & 1u, nullptr)) atomicOr(a.err, PKD_DEV_ERR_TIMEOUT);
      }
    }
  }
}

// ---------------------------------------------------------------- consumers
template <int G>
struct Shape {
  static constexpr int J = (G == 8) ? 4 : 8;   // token steps per batch (per half-warp)
  static constexpr int NB = (kTS / 2) / J;     // batches per stage
  static constexpr int N0 = G * J;             // partials per lane before the reduce
  static constexpr int E = (N0 >= 16) ? N0 / 16 : 1;  // scores per lane after it
  // li bits that index tokens within a head's lane group (the others index
  // the head).  For G = 1 the lowest bit is a duplicate, left out.
  static constexpr int TOKBITS = (G == 1) ? 14 : (16 / G - 1);
};

template <int G, int kRing>
__device__ void run_consumer_fma(const DecodeArgs& a, int it0, int it1, const uint8_t* stages,
                             int stage_bytes, uint64_t* full, uint64_t* empty,
                             volatile int* abort_flag, float* pbuf, float* sbuf, int warp,
                             int lane) {
  using S = Shape<G>;
  constexpr int J = S::J, NB = S::NB, N0 = S::N0, E = S::E;
  const int hk = warp;
  const int hw = lane >> 4;
  const int li = lane & 15;
  const int rs = rows_tok_stride(a);

  // Which (head, step) values this lane holds after the reduce-scatter.
  int vbase = 0;
  {
    int n = N0;
    const int masks[4] = {8, 4, 2, 1};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if (n > 1) {
        n >>= 1;
        if (li & masks[k]) vbase += n;
      }
    }
  }
  const int my_head = vbase / J;
  const bool leader = ((li & S::TOKBITS) == 0) && hw == 0;

  pdl_wait();   // q may come from the previous kernel in the stream
  uint32_t stage = 0;
  for (int it = it0; it < it1; ++it) {
    const int32_t* item = a.sched + a.off_items + (int64_t)it * kItemWords;
    const int req = item[0], tb = item[1], te = item[2], dst = item[3];

    // q of this KV head's group, pre-scaled by log2(e)/sqrt(D).
    float qf[G][8];
    {
      const uint16_t* qp = a.q + ((int64_t)req * a.hq + (int64_t)hk * G) * kHeadDim + 8 * li;
#pragma unroll
      for (int i = 0; i < G; ++i) {
        const uint4 r = __ldg(reinterpret_cast<const uint4*>(qp + (int64_t)i * kHeadDim));
        bf16x8_to_f32(r, qf[i]);
#pragma unroll
        for (int d = 0; d < 8; ++d) qf[i][d] *= a.scale_log2;
      }
    }
    float acc[G][8];
#pragma unroll
    for (int i = 0; i < G; ++i)
#pragma unroll
      for (int d = 0; d < 8; ++d) acc[i][d] = 0.f;
    float m_run = -CUDART_INF_F;  // running max (log2 units) of my_head
    float l_run = 0.f;            // this lane's share of the running sum

    for (int t = tb; t < te; t += kTS) {
      const int n = min(kTS, te - t);
      const int slot = (int)(stage % kRing);
      const bool got = mbar_wait(&full[slot], (stage / kRing) & 1u, abort_flag);
      if (!__all_sync(kFull, got)) {
        if (lane == 0) raise_error(a.err, abort_flag, PKD_DEV_ERR_TIMEOUT);
        return;
      }
      const uint8_t* ks = stages + (size_t)slot * stage_bytes + hk * (kHeadDim * 2) + li * 16;
      const uint8_t* vs = ks + rows_v_base(a, kTS);

#pragma unroll
      for (int b = 0; b < NB; ++b) {
        if (2 * b * J >= n) break;
        // ---- scores: partial dot products over this lane's 8 dims
        float part[N0];
#pragma unroll
        for (int j = 0; j < J; ++j) {
          const int tok = 2 * (b * J + j) + hw;
          float k8[8];
          bf16x8_to_f32(*reinterpret_cast<const uint4*>(ks + (size_t)tok * rs), k8);
#pragma unroll
          for (int i = 0; i < G; ++i) {
            float s = 0.f;
#pragma unroll
            for (int d = 0; d < 8; ++d) s = fmaf(qf[i][d], k8[d], s);
            part[i * J + j] = s;
          }
        }
        // ---- reduce-scatter across the 16 lanes of the half-warp
        float sv[E];
        {
          float r1[N0 / 2];
          rs_level<N0>(part, r1, 8, (li & 8) != 0);
          float r2[N0 / 4];
          rs_level<N0 / 2>(r1, r2, 4, (li & 4) != 0);
          float r3[N0 / 8];
          rs_level<N0 / 4>(r2, r3, 2, (li & 2) != 0);
          if constexpr (N0 >= 16) {
            float r4[N0 / 16];
            rs_level<N0 / 8>(r3, r4, 1, (li & 1) != 0);
#pragma unroll
            for (int e = 0; e < E; ++e) sv[e] = r4[e];
          } else {
            sv[0] = r3[0] + __shfl_xor_sync(kFull, r3[0], 1);
          }
        }
        // ---- online softmax for my_head over this batch's tokens
        float mx = -CUDART_INF_F;
        int toks[E];
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const int j = (vbase + e) % J;
          toks[e] = 2 * (b * J + j) + hw;
          if (toks[e] >= n) sv[e] = -CUDART_INF_F;
          mx = fmaxf(mx, sv[e]);
        }
#pragma unroll
        for (int mask = 1; mask < 16; mask <<= 1)
          if (S::TOKBITS & mask) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, mask));
        mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 16));
        const float m_new = fmaxf(m_run, mx);
        const float m_use = (m_new == -CUDART_INF_F) ? 0.f : m_new;
        const float alpha = exp2f(m_run - m_use);
        float psum = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const float p = exp2f(sv[e] - m_use);
          psum += p;
          pbuf[toks[e] * G + my_head] = p;
        }
        l_run = l_run * alpha + psum;
        m_run = m_new;
        if (leader) sbuf[my_head] = alpha;
        __syncwarp();
        // ---- rescale and accumulate P.V over this lane's dims
#pragma unroll
        for (int i = 0; i < G; ++i) {
          const float al = sbuf[i];
#pragma unroll
          for (int d = 0; d < 8; ++d) acc[i][d] *= al;
        }
#pragma unroll
        for (int j = 0; j < J; ++j) {
          const int tok = 2 * (b * J + j) + hw;
          const int src_row = (tok < n) ? tok : 0;   // p = 0 there; row 0 is valid
          float p[G];
          if constexpr (G == 8) {
            const float4 p0 = *reinterpret_cast<const float4*>(pbuf + tok * G);
            const float4 p1 = *reinterpret_cast<const float4*>(pbuf + tok * G + 4);
            p[0] = p0.x; p[1] = p0.y; p[2] = p0.z; p[3] = p0.w;
            p[4] = p1.x; p[5] = p1.y; p[6] = p1.z; p[7] = p1.w;
          } else if constexpr (G == 4) {
            const float4 p0 = *reinterpret_cast<const float4*>(pbuf + tok * G);
            p[0] = p0.x; p[1] = p0.y; p[2] = p0.z; p[3] = p0.w;
          } else if constexpr (G == 2) {
            const float2 p0 = *reinterpret_cast<const float2*>(pbuf + tok * G);
            p[0] = p0.x; p[1] = p0.y;
          } else {
            p[0] = pbuf[tok];
          }
          float v8[8];
          bf16x8_to_f32(*reinterpret_cast<const uint4*>(vs + (size_t)src_row * rs), v8);
#pragma unroll
          for (int i = 0; i < G; ++i)
#pragma unroll
            for (int d = 0; d < 8; ++d) acc[i][d] = fmaf(p[i], v8[d], acc[i][d]);
        }
        __syncwarp();
      }
      if (lane == 0) mbar_arrive(&empty[slot]);
      ++stage;
    }

    // ---- epilogue: combine half-warps, normalise, write
#pragma unroll
    for (int i = 0; i < G; ++i)
#pragma unroll
      for (int d = 0; d < 8; ++d) acc[i][d] += __shfl_xor_sync(kFull, acc[i][d], 16);
    float l = l_run;
#pragma unroll
    for (int mask = 1; mask < 16; mask <<= 1)
      if (S::TOKBITS & mask) l += __shfl_xor_sync(kFull, l, mask);
    l += __shfl_xor_sync(kFull, l, 16);
    if (leader) {
      sbuf[8 + my_head] = m_run;
      sbuf[16 + my_head] = l;
    }
    __syncwarp();
#pragma unroll
    for (int i = 0; i < G; ++i) {
      if (G > 1 ? ((i & 1) != hw) : (hw != 0)) continue;
      const float m = sbuf[8 + i];
      const float lsum = sbuf[16 + i];
      const float inv = a.v_scale / lsum;
      const float lse_nat = (m + log2f(lsum)) * 0.69314718055994530942f;
      const int64_t qrow = (int64_t)req * a.hq + (int64_t)hk * G + i;
      if (dst < 0) {
        uint32_t w[4];
#pragma unroll
        for (int d = 0; d < 4; ++d)
          w[d] = f32_to_bf16_rne(acc[i][2 * d] * inv) |
                 (f32_to_bf16_rne(acc[i][2 * d + 1] * inv) << 16);
        *reinterpret_cast<uint4*>(a.out + qrow * kHeadDim + 8 * li) =
            make_uint4(w[0], w[1], w[2], w[3]);
        if (a.lse != nullptr && li == 0) a.lse[qrow] = lse_nat;
      } else {
        const int64_t prow = (int64_t)dst * a.hq + (int64_t)hk * G + i;
        float4* o = reinterpret_cast<float4*>(a.o_part + prow * kHeadDim + 8 * li);
        o[0] = make_float4(acc[i][0] * inv, acc[i][1] * inv, acc[i][2] * inv, acc[i][3] * inv);
        o[1] = make_float4(acc[i][4] * inv, acc[i][5] * inv, acc[i][6] * inv, acc[i][7] * inv);
        if (li == 0) a.l_part[prow] = lse_nat;
      }
    }
    __syncwarp();
  }
}


// ------------------------------------------------- tensor-core consumer (MMA)
// The GQA group as a thin matrix: S = Q K^T with the group's G query heads
// as the 16-row M dimension (rows >= G are zero), 8 tokens per N tile and 16
// dims per K step (mma.sync m16n8k16, bf16 in, fp32 accumulate); then
// O += P V with P taken straight from the S accumulators (converted to bf16)
// and V fragments loaded transposed with ldmatrix.  One K/V read from shared
// memory serves the whole group.  Softmax statistics stay in fp32.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                          uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// D = A B + D with A 16x16 whose rows 8..15 are zero (a1 = a3 = 0), B 16x8,
// fp32 accumulate.  Only rows 0..7 (d0, d1) are kept: the group has <= 8
// query heads, so the other half of the tile is always zero.
__device__ __forceinline__ void mma_bf16(float (&d)[2], uint32_t a0, uint32_t a2, uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "{\n\t.reg .f32 z0, z1;\n\t"
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,z0,z1}, {%2,%3,%4,%5}, "
      "{%6,%7}, {%8,%9,%10,%10};\n\t}"
      : "=f"(d[0]), "=f"(d[1])
      : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1), "f"(d[0]), "f"(d[1]), "f"(0.f));
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  return f32_to_bf16_rne(lo) | (f32_to_bf16_rne(hi) << 16);
}

// Shared-memory addresses of KV head hk's ldmatrix rows in a 16-token bf16
// stage.  K (no transpose), for N tile nt and K-step pair kp: lane L gives
// token 8 nt + L % 8, 16-byte chunk 4 kp + L / 8 of the head's 256 bytes.
// V (transposed), for dim pair dp: token (L / 8 & 1) * 8 + L % 8, chunk
// 2 dp + L / 16.
//  * token rows: K row of token t at t * rs, V row at v_base + t * rs (see
//    rows_tok_stride), head at hk * 256;
//  * page tiles: K box at 0, V box at 16 * row_bytes; inside a box the
//    128-byte line (2 hk + chunk / 8) * 16 + t holds the chunk at position
//    (chunk % 8) ^ (t % 8).
template <bool kTiles>
struct Bf16Frags {
  uint32_t k, v, kx, vx;
  int rs, vz;   // token-row stride; V rows' base (token rows)
  __device__ __forceinline__ Bf16Frags(const DecodeArgs& a, int hk, int lane) {
    vz = 0;
    rs = rows_tok_stride(a);
    const int r = lane & 7;
    if constexpr (kTiles) {
      k = (uint32_t)((hk * 32 + r) * 128);
      kx = (uint32_t)(((lane >> 3) ^ r) << 4);
      v = (uint32_t)(16 * a.row_bytes + (hk * 32 + ((lane >> 3) & 1) * 8 + r) * 128);
      vx = (uint32_t)(((lane >> 4) ^ r) << 4);
    } else {
      k = (uint32_t)(r * rs + hk * (kHeadDim * 2) + (lane >> 3) * 16);
      v = (uint32_t)(rows_v_base(a, kTS) + (((lane >> 3) & 1) * 8 + r) * rs +
                     hk * (kHeadDim * 2) + (lane >> 4) * 16);
      kx = vx = 0;
      vz = rows_v_base(a, kTS);
    }
  }
  __device__ __forceinline__ uint32_t kaddr(uint32_t sbase, int nt, int kp) const {
    if constexpr (kTiles)
      return sbase + k + (uint32_t)((kp >> 1) * 2048 + nt * 1024) + (kx ^ (uint32_t)((kp & 1) << 6));
    else
      return sbase + k + (uint32_t)(nt * 8 * rs + kp * 64);
  }
  __device__ __forceinline__ uint32_t vaddr(uint32_t sbase, int dp) const {
    if constexpr (kTiles)
      return sbase + v + (uint32_t)((dp >> 2) * 2048) + (vx ^ (uint32_t)((dp & 3) << 5));
    else
      return sbase + v + (uint32_t)(dp * 32);
  }
  // Zero head hk's V tokens n .. 15 of the stage (stale or past-the-end
  // bytes: P = 0 there, but 0 x NaN would poison O).
  __device__ __forceinline__ void zero_v_tail(uint8_t* stage, int row_bytes, int hk, int lane,
                                              int n) const {
    if constexpr (kTiles) {
      uint8_t* z = stage + 16 * row_bytes + (hk * 32 + ((lane >> 3) & 1) * 16) * 128 + (lane & 7) * 16;
      for (int r = n + (lane >> 4); r < kTS; r += 2)
        *reinterpret_cast<uint4*>(z + r * 128) = make_uint4(0, 0, 0, 0);
    } else {
      uint8_t* z = stage + vz + hk * (kHeadDim * 2) + (lane & 15) * 16;
      for (int r = n + (lane >> 4); r < kTS; r += 2)
        *reinterpret_cast<uint4*>(z + (size_t)r * rs) = make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
    __syncwarp();
  }
};

// A fragments of the group's queries: row = query head grp, two bf16 per
// register (dims 16 ks + 2 tig, +1 and the same + 8).
template <int G>
__device__ __forceinline__ void load_q_frags(const DecodeArgs& a, int req, int hk, int grp,
                                             int tig, bool row_ok, uint32_t (&qa0)[8],
                                             uint32_t (&qa2)[8]) {
  const uint32_t* qp = reinterpret_cast<const uint32_t*>(
      a.q + ((int64_t)req * a.hq + (int64_t)hk * G + (row_ok ? grp : 0)) * kHeadDim);
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    qa0[ks] = row_ok ? __ldg(qp + ks * 8 + tig) : 0u;
    qa2[ks] = row_ok ? __ldg(qp + ks * 8 + 4 + tig) : 0u;
  }
}

template <int G, bool kTiles, int kRing>
__device__ void run_consumer_mma(const DecodeArgs& a, int it0, int it1, const uint8_t* stages,
                                 int stage_bytes, uint64_t* full, uint64_t* empty,
                                 volatile int* abort_flag, int warp, int lane) {
  const int hk = warp;
  const int grp = lane >> 2;   // fragment row: query head within the group
  const int tig = lane & 3;    // fragment column pair
  const bool row_ok = grp < G;
  const uint32_t stage0 = smem_u32(stages);
  const Bf16Frags<kTiles> fr(a, hk, lane);

  // the item and its queries are fetched one item ahead
  const int32_t* item = a.sched + a.off_items + (int64_t)it0 * kItemWords;
  int req = item[0], tb = item[1], te = item[2], dst = item[3];
  // q is read at once, like the KV cache; the first write (outputs or the
  // partial states the previous kernel may still read) waits for it
  bool waited = false;
  uint32_t qa0[8], qa2[8];
  load_q_frags<G>(a, req, hk, grp, tig, row_ok, qa0, qa2);

  uint32_t stage = 0;
  for (int it = it0; it < it1; ++it) {
    int n_req = 0, n_tb = 0, n_te = 0, n_dst = -1;
    uint32_t nq0[8], nq2[8];
    if (it + 1 < it1) {
      const int32_t* nx = a.sched + a.off_items + (int64_t)(it + 1) * kItemWords;
      n_req = nx[0];
      n_tb = nx[1];
      n_te = nx[2];
      n_dst = nx[3];
      load_q_frags<G>(a, n_req, hk, grp, tig, row_ok, nq0, nq2);
    }
    float o[16][2];
#pragma unroll
    for (int dt = 0; dt < 16; ++dt) o[dt][0] = o[dt][1] = 0.f;
    float m_run = -CUDART_INF_F;
    float l_run = 0.f;

    for (int t = tb; t < te; t += kTS) {
      const int n = min(kTS, te - t);
      const int slot = (int)(stage % kRing);
      const bool got = mbar_wait(&full[slot], (stage / kRing) & 1u, abort_flag);
      if (!__all_sync(kFull, got)) {
        if (lane == 0) raise_error(a.err, abort_flag, PKD_DEV_ERR_TIMEOUT);
        if (!waited) pdl_wait();   // complete only after the previous kernel
        return;
      }
      const uint32_t sbase = stage0 + (uint32_t)(slot * stage_bytes);
      if (n < kTS)
        fr.zero_v_tail(const_cast<uint8_t*>(stages) + (size_t)slot * stage_bytes, a.row_bytes, hk,
                       lane, n);
      // ---- S = Q K^T for two 8-token tiles
      float sc[2][2];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        sc[nt][0] = sc[nt][1] = 0.f;
#pragma unroll
        for (int kp = 0; kp < 4; ++kp) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(fr.kaddr(sbase, nt, kp), b0, b1, b2, b3);
          mma_bf16(sc[nt], qa0[2 * kp], qa2[2 * kp], b0, b1);
          mma_bf16(sc[nt], qa0[2 * kp + 1], qa2[2 * kp + 1], b2, b3);
        }
      }
      // ---- online softmax on this lane's row (query head grp), 4 tokens
      float s4[4];
      float mx = -CUDART_INF_F;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int tok = nt * 8 + 2 * tig + c;
          const float v = (tok < n) ? sc[nt][c] * a.scale_log2 : -CUDART_INF_F;
          s4[nt * 2 + c] = v;
          mx = fmaxf(mx, v);
        }
      mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
      const float m_new = fmaxf(m_run, mx);
      const float m_use = (m_new == -CUDART_INF_F) ? 0.f : m_new;
      const float alpha = exp2f(m_run - m_use);
      float p4[4];
      float psum = 0.f;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        p4[k] = exp2f(s4[k] - m_use);
        psum += p4[k];
      }
      l_run = l_run * alpha + psum;
      m_run = m_new;
      const uint32_t pa0 = pack_bf16x2(p4[0], p4[1]);   // tokens 2 tig, 2 tig + 1
      const uint32_t pa2 = pack_bf16x2(p4[2], p4[3]);   // tokens 8 + 2 tig, 9 + 2 tig
      // ---- O = alpha O + P V over 16 dim tiles
#pragma unroll
      for (int dp = 0; dp < 8; ++dp) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(fr.vaddr(sbase, dp), b0, b1, b2, b3);
        o[2 * dp][0] *= alpha;
        o[2 * dp][1] *= alpha;
        o[2 * dp + 1][0] *= alpha;
        o[2 * dp + 1][1] *= alpha;
        mma_bf16(o[2 * dp], pa0, pa2, b0, b1);
        mma_bf16(o[2 * dp + 1], pa0, pa2, b2, b3);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
      ++stage;
    }

    // ---- epilogue: row sums over the quad, normalise, write
    float l = l_run;
    l += __shfl_xor_sync(kFull, l, 1);
    l += __shfl_xor_sync(kFull, l, 2);
    if (!waited) {
      pdl_wait();
      waited = true;
    }
    if (row_ok) {
      const float inv = a.v_scale / l;
      const float lse_nat = (m_run + log2f(l)) * 0.69314718055994530942f;
      const int64_t qrow = (int64_t)req * a.hq + (int64_t)hk * G + grp;
      if (dst < 0) {
        uint32_t* op = reinterpret_cast<uint32_t*>(a.out + qrow * kHeadDim) + tig;
#pragma unroll
        for (int dt = 0; dt < 16; ++dt) op[dt * 4] = pack_bf16x2(o[dt][0] * inv, o[dt][1] * inv);
        if (a.lse != nullptr && tig == 0) a.lse[qrow] = lse_nat;
      } else {
        const int64_t prow = (int64_t)dst * a.hq + (int64_t)hk * G + grp;
        float2* op = reinterpret_cast<float2*>(a.o_part + prow * kHeadDim) + tig;
#pragma unroll
        for (int dt = 0; dt < 16; ++dt) op[dt * 4] = make_float2(o[dt][0] * inv, o[dt][1] * inv);
        if (tig == 0) a.l_part[prow] = lse_nat;
      }
    }
    if (it + 1 < it1) {
      req = n_req;
      tb = n_tb;
      te = n_te;
      dst = n_dst;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        qa0[ks] = nq0[ks];
        qa2[ks] = nq2[ks];
      }
    }
  }
}


// --------------------------------------- shared-prefix row-block consumer (MMA)
// A work item covers a block of n_req <= 16 / G consecutive requests that
// attend over the same pages (a shared prefix: FlashInfer 完全拆解, Composable
// Format, the (R, 1) block).  All 16 rows of the m16n8k16 tile are used:
// row r is request r / G of the block and query head hk * G + r % G, so one
// K/V read from shared memory serves n_req * G query rows.
__device__ __forceinline__ void mma_bf16_full(float (&d)[4], uint32_t a0, uint32_t a1,
                                              uint32_t a2, uint32_t a3, uint32_t b0,
                                              uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// One tile row's online-softmax update over this lane's 4 scores (tokens
// 2 tig, 2 tig + 1, 8 + 2 tig, 9 + 2 tig); returns the rescale factor.
__device__ __forceinline__ float softmax_row(float (&s4)[4], float& m_run, float& l_run) {
  float mx = fmaxf(fmaxf(s4[0], s4[1]), fmaxf(s4[2], s4[3]));
  mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
  const float m_new = fmaxf(m_run, mx);
  const float m_use = (m_new == -CUDART_INF_F) ? 0.f : m_new;
  const float alpha = exp2f(m_run - m_use);
  float psum = 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    s4[k] = exp2f(s4[k] - m_use);
    psum += s4[k];
  }
  l_run = l_run * alpha + psum;
  m_run = m_new;
  return alpha;
}

template <int G, bool kTiles, int kRing>
__device__ void run_consumer_mma_block(const DecodeArgs& a, int it0, int it1,
                                       const uint8_t* stages, int stage_bytes, uint64_t* full,
                                       uint64_t* empty, volatile int* abort_flag, int warp,
                                       int lane) {
  const int hk = warp;
  const int grp = lane >> 2;
  const int tig = lane & 3;
  // the lane's two tile rows: grp and grp + 8
  const int rq0 = grp / G, hd0 = grp % G;
  const int rq1 = (grp + 8) / G, hd1 = (grp + 8) % G;
  const uint32_t stage0 = smem_u32(stages);
  const Bf16Frags<kTiles> fr(a, hk, lane);
  pdl_wait();   // q may come from the previous kernel in the stream
  uint32_t stage = 0;
  for (int it = it0; it < it1; ++it) {
    const int32_t* item = a.sched + a.off_items + (int64_t)it * kItemWords;
    const int req = item[0], tb = item[1], te = item[2], dst = item[3];
    const int n_req = item[5], stride = item[6];
    const bool ok0 = rq0 < n_req, ok1 = rq1 < n_req;
    uint32_t qa0[8], qa1[8], qa2[8], qa3[8];
    {
      const uint32_t* q0 = reinterpret_cast<const uint32_t*>(
          a.q + ((int64_t)(req + (ok0 ? rq0 : 0)) * a.hq + (int64_t)hk * G + hd0) * kHeadDim);
      const uint32_t* q1 = reinterpret_cast<const uint32_t*>(
          a.q + ((int64_t)(req + (ok1 ? rq1 : 0)) * a.hq + (int64_t)hk * G + hd1) * kHeadDim);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        qa0[ks] = ok0 ? __ldg(q0 + ks * 8 + tig) : 0u;
        qa2[ks] = ok0 ? __ldg(q0 + ks * 8 + 4 + tig) : 0u;
        qa1[ks] = ok1 ? __ldg(q1 + ks * 8 + tig) : 0u;
        qa3[ks] = ok1 ? __ldg(q1 + ks * 8 + 4 + tig) : 0u;
      }
    }
    float o[16][4];
#pragma unroll
    for (int dt = 0; dt < 16; ++dt)
#pragma unroll
      for (int c = 0; c < 4; ++c) o[dt][c] = 0.f;
    float m0 = -CUDART_INF_F, m1 = -CUDART_INF_F, l0 = 0.f, l1 = 0.f;

    for (int t = tb; t < te; t += kTS) {
      const int n = min(kTS, te - t);
      const int slot = (int)(stage % kRing);
      const bool got = mbar_wait(&full[slot], (stage / kRing) & 1u, abort_flag);
      if (!__all_sync(kFull, got)) {
        if (lane == 0) raise_error(a.err, abort_flag, PKD_DEV_ERR_TIMEOUT);
        return;
      }
      const uint32_t sbase = stage0 + (uint32_t)(slot * stage_bytes);
      if (n < kTS)
        fr.zero_v_tail(const_cast<uint8_t*>(stages) + (size_t)slot * stage_bytes, a.row_bytes, hk,
                       lane, n);
      // S = Q K^T as four independent MMA chains (N tile x K-step parity),
      // summed at the end: the tile is all 16 rows, so chain latency, not
      // issue, bounds a single chain
      float sc[2][4], sx[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int c = 0; c < 4; ++c) sc[nt][c] = sx[nt][c] = 0.f;
#pragma unroll
      for (int kp = 0; kp < 4; ++kp) {
        uint32_t b[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
          ldsm_x4(fr.kaddr(sbase, nt, kp), b[nt][0], b[nt][1], b[nt][2], b[nt][3]);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
          mma_bf16_full(sc[nt], qa0[2 * kp], qa1[2 * kp], qa2[2 * kp], qa3[2 * kp], b[nt][0],
                        b[nt][1]);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
          mma_bf16_full(sx[nt], qa0[2 * kp + 1], qa1[2 * kp + 1], qa2[2 * kp + 1],
                        qa3[2 * kp + 1], b[nt][2], b[nt][3]);
      }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int c = 0; c < 4; ++c) sc[nt][c] += sx[nt][c];
      float s0[4], s1[4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const bool v = nt * 8 + 2 * tig + c < n;
          s0[nt * 2 + c] = v ? sc[nt][c] * a.scale_log2 : -CUDART_INF_F;
          s1[nt * 2 + c] = v ? sc[nt][2 + c] * a.scale_log2 : -CUDART_INF_F;
        }
      const float al0 = softmax_row(s0, m0, l0);
      const float al1 = softmax_row(s1, m1, l1);
      const uint32_t pa0 = pack_bf16x2(s0[0], s0[1]);   // row grp, tokens 2 tig, +1
      const uint32_t pa1 = pack_bf16x2(s1[0], s1[1]);   // row grp + 8
      const uint32_t pa2 = pack_bf16x2(s0[2], s0[3]);   // row grp, tokens 8 + 2 tig, +1
      const uint32_t pa3 = pack_bf16x2(s1[2], s1[3]);   // row grp + 8
#pragma unroll
      for (int dp = 0; dp < 8; ++dp) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(fr.vaddr(sbase, dp), b0, b1, b2, b3);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          o[2 * dp + h][0] *= al0;
          o[2 * dp + h][1] *= al0;
          o[2 * dp + h][2] *= al1;
          o[2 * dp + h][3] *= al1;
        }
        mma_bf16_full(o[2 * dp], pa0, pa1, pa2, pa3, b0, b1);
        mma_bf16_full(o[2 * dp + 1], pa0, pa1, pa2, pa3, b2, b3);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
      ++stage;
    }

    l0 += __shfl_xor_sync(kFull, l0, 1);
    l0 += __shfl_xor_sync(kFull, l0, 2);
    l1 += __shfl_xor_sync(kFull, l1, 1);
    l1 += __shfl_xor_sync(kFull, l1, 2);
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const bool ok = rr ? ok1 : ok0;
      if (!ok) continue;
      const int rq = rr ? rq1 : rq0;
      const int head = hk * G + (rr ? hd1 : hd0);
      const float l = rr ? l1 : l0;
      const float m = rr ? m1 : m0;
      const float inv = a.v_scale / l;
      const float lse_nat = (m + log2f(l)) * 0.69314718055994530942f;
      if (dst < 0) {
        const int64_t qrow = (int64_t)(req + rq) * a.hq + head;
        uint32_t* op = reinterpret_cast<uint32_t*>(a.out + qrow * kHeadDim) + tig;
#pragma unroll
        for (int dt = 0; dt < 16; ++dt)
          op[dt * 4] = pack_bf16x2(o[dt][2 * rr] * inv, o[dt][2 * rr + 1] * inv);
        if (a.lse != nullptr && tig == 0) a.lse[qrow] = lse_nat;
      } else {
        const int64_t prow = (int64_t)(dst + rq * stride) * a.hq + head;
        float2* op = reinterpret_cast<float2*>(a.o_part + prow * kHeadDim) + tig;
#pragma unroll
        for (int dt = 0; dt < 16; ++dt)
          op[dt * 4] = make_float2(o[dt][2 * rr] * inv, o[dt][2 * rr + 1] * inv);
        if (tig == 0) a.l_part[prow] = lse_nat;
      }
    }
  }
}


// ------------------------------------------------------ FP8-E4M3 KV consumer
// The cache holds e4m3 (one byte per element: half the bytes per token);
// k_scale and v_scale are folded into the score scale and the output.  The
// e4m3 bytes go straight from the shared-memory stage into f16 MMA
// fragments -- every e4m3 value is an f16, cvt.f16x2.e4m3x2 is exact:
//  * K: ldmatrix on the byte rows gives each lane 4 consecutive dims of one
//    token; in the MMA's K (dims) order, k = 2t, 2t+1, 2t+8, 2t+9 stand for
//    dims 4t .. 4t+3 of each 16-dim block, and q's A fragments are loaded in
//    the same order, so the dot products are unchanged;
//  * V: ldmatrix.trans on the byte rows gives each lane 2 tokens x 2 adjacent
//    dims; one byte permute and two converts make the B fragments of two
//    N tiles (even and odd dims of the block), so the lane ends with 4
//    consecutive output dims per block.
// q is scaled per row into [-1, 1] (no f16 overflow whatever the bf16 range)
// and the factor folded into the score scale; P is f16.  A stage holds 32
// tokens (the same bytes as 16 bf16 tokens), folded in one softmax update.
constexpr int kFp8Tokens = 32;

__device__ __forceinline__ void mma_f16(float (&d)[2], uint32_t a0, uint32_t a2, uint32_t b0,
                                        uint32_t b1) {
  asm volatile(
      "{\n\t.reg .f32 z0, z1;\n\t"
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,z0,z1}, {%2,%3,%4,%5}, "
      "{%6,%7}, {%8,%9,%10,%10};\n\t}"
      : "=f"(d[0]), "=f"(d[1])
      : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1), "f"(d[0]), "f"(d[1]), "f"(0.f));
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Four e4m3 bytes -> two f16x2 (bytes 0, 1 -> lo; bytes 2, 3 -> hi); every
// e4m3 value is exact in f16.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t r, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(r));
}

// Shared-memory addresses of KV head hk's ldmatrix rows in a 32-token e4m3
// stage (16-token tile st).  K, for N tile nt and x4 kq: lane L gives token
// 16 st + 8 nt + L % 8, 16-byte chunk 4 kq + L / 8 of the head's 128 bytes.
// V (trans), for x4 vp: token 16 st + (L / 8 & 1) * 8 + L % 8, chunk
// 2 vp + L / 16.
//  * token rows: K row of token t at t * rs, V row at v_base + t * rs (see
//    rows_tok_stride), head at hk * 128;
//  * page tiles: K box st at st * box, V box st at (2 + st) * box (box =
//    16 * row_bytes); inside a box the line hk * 16 + t holds chunk c at
//    position c ^ (t % 8).
template <bool kTiles>
struct Fp8Frags {
  uint32_t k, v, kx, vx, box;
  int rs, vz;   // token-row stride; V rows' base (token rows)
  __device__ __forceinline__ Fp8Frags(const DecodeArgs& a, int hk, int lane) {
    rs = rows_tok_stride(a);
    vz = 0;
    box = (uint32_t)(16 * a.row_bytes);
    const int r = lane & 7;
    if constexpr (kTiles) {
      k = (uint32_t)((hk * 16 + r) * 128);
      kx = (uint32_t)(((lane >> 3) ^ r) << 4);
      v = 2 * box + (uint32_t)((hk * 16 + ((lane >> 3) & 1) * 8 + r) * 128);
      vx = (uint32_t)(((lane >> 4) ^ r) << 4);
    } else {
      k = (uint32_t)(r * rs + hk * kHeadDim + (lane >> 3) * 16);
      v = (uint32_t)(rows_v_base(a, kFp8Tokens) + (((lane >> 3) & 1) * 8 + r) * rs +
                     hk * kHeadDim + (lane >> 4) * 16);
      kx = vx = 0;
      vz = rows_v_base(a, kFp8Tokens);
    }
  }
  __device__ __forceinline__ uint32_t kaddr(uint32_t sbase, int st, int nt, int kq) const {
    if constexpr (kTiles)
      return sbase + (uint32_t)st * box + k + (uint32_t)(nt * 1024) + (kx ^ (uint32_t)(kq << 6));
    else
      return sbase + k + (uint32_t)((st * 16 + nt * 8) * rs + kq * 64);
  }
  __device__ __forceinline__ uint32_t vaddr(uint32_t sbase, int st, int vp) const {
    if constexpr (kTiles)
      return sbase + (uint32_t)st * box + v + (vx ^ (uint32_t)(vp << 5));
    else
      return sbase + v + (uint32_t)(st * 16 * rs + vp * 32);
  }
  // Zero head hk's V tokens n .. (end of the copied rows) of the stage
  // (0x7f / 0xff bytes are NaN in e4m3).
  __device__ __forceinline__ void zero_v_tail(uint8_t* stage, int hk, int lane, int n) const {
    if constexpr (kTiles) {
      const int end = (n + 15) & ~15;   // the copied boxes
      uint8_t* z = stage + 2 * box + hk * 16 * 128 + (lane & 7) * 16;
      for (int r = n + (lane >> 3); r < end; r += 4)
        *reinterpret_cast<uint4*>(z + (r >> 4) * box + (r & 15) * 128) = make_uint4(0, 0, 0, 0);
    } else {
      uint8_t* z = stage + vz + hk * kHeadDim + (lane & 7) * 16;
      for (int r = n + (lane >> 3); r < kFp8Tokens; r += 4)
        *reinterpret_cast<uint4*>(z + (size_t)r * rs) = make_uint4(0, 0, 0, 0);
    }
    fence_proxy_async_smem();
    __syncwarp();
  }
};

// One stage folded into the running state: kNt 8-token N tiles (4: both
// 16-token halves of the stage; 2: the first half only, when the stage holds
// <= 16 tokens -- the second half was not copied).  The S accumulators form kNt
// independent MMA chains; one softmax update and one rescale of O per stage.
template <int kNt, bool kTiles>
__device__ __forceinline__ void fp8_stage(const Fp8Frags<kTiles>& fr, uint32_t sbase, int n,
                                          int tig, const uint32_t (&qa0)[8],
                                          const uint32_t (&qa2)[8], float s_scale,
                                          float (&oe)[8][2], float (&oo)[8][2], float& m_run,
                                          float& l_run) {
  // ---- S = Q K^T
  float sc[kNt][2];
#pragma unroll
  for (int nt = 0; nt < kNt; ++nt) sc[nt][0] = sc[nt][1] = 0.f;
#pragma unroll
  for (int kq = 0; kq < 2; ++kq) {
    uint32_t r[kNt][4];
#pragma unroll
    for (int nt = 0; nt < kNt; ++nt)
      ldsm_x4(fr.kaddr(sbase, nt >> 1, nt & 1, kq), r[nt][0], r[nt][1], r[nt][2], r[nt][3]);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
#pragma unroll
      for (int nt = 0; nt < kNt; ++nt) {
        uint32_t b0, b1;
        e4m3x4_to_f16x2x2(r[nt][j], b0, b1);
        mma_f16(sc[nt], qa0[kq * 4 + j], qa2[kq * 4 + j], b0, b1);
      }
    }
  }
  // ---- online softmax over this lane's 2 kNt scores (query head grp)
  float mx = -CUDART_INF_F;
#pragma unroll
  for (int nt = 0; nt < kNt; ++nt)
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int tok = nt * 8 + 2 * tig + c;
      sc[nt][c] = (tok < n) ? sc[nt][c] * s_scale : -CUDART_INF_F;
      mx = fmaxf(mx, sc[nt][c]);
    }
  mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
  const float m_new = fmaxf(m_run, mx);
  const float m_use = (m_new == -CUDART_INF_F) ? 0.f : m_new;
  const float alpha = exp2f(m_run - m_use);
  float psum = 0.f;
#pragma unroll
  for (int nt = 0; nt < kNt; ++nt)
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      sc[nt][c] = exp2f(sc[nt][c] - m_use);
      psum += sc[nt][c];
    }
  l_run = l_run * alpha + psum;
  m_run = m_new;
  // P as A fragments, one pair per 16-token K step st
  uint32_t pa0[kNt / 2], pa2[kNt / 2];
#pragma unroll
  for (int st = 0; st < kNt / 2; ++st) {
    pa0[st] = pack_f16x2(sc[2 * st][0], sc[2 * st][1]);          // tokens 16 st + 2 tig, +1
    pa2[st] = pack_f16x2(sc[2 * st + 1][0], sc[2 * st + 1][1]);  // 16 st + 8 + 2 tig, +1
  }
#pragma unroll
  for (int vb = 0; vb < 8; ++vb) {
    oe[vb][0] *= alpha;
    oe[vb][1] *= alpha;
    oo[vb][0] *= alpha;
    oo[vb][1] *= alpha;
  }
  // ---- O += P V: per x4.trans, dim blocks 2 vp and 2 vp + 1
#pragma unroll
  for (int vp = 0; vp < 4; ++vp) {
#pragma unroll
    for (int st = 0; st < kNt / 2; ++st) {
      uint32_t r[4];
      ldsm_x4_t(fr.vaddr(sbase, st, vp), r[0], r[1], r[2], r[3]);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int vb = 2 * vp + h;
        // r[2h]: tokens 2 tig, 2 tig + 1; r[2h + 1]: tokens 8 + 2 tig, 9 + 2 tig
        uint32_t e0, o0, e1, o1;
        e4m3x4_to_f16x2x2(__byte_perm(r[2 * h], 0u, 0x3120), e0, o0);
        e4m3x4_to_f16x2x2(__byte_perm(r[2 * h + 1], 0u, 0x3120), e1, o1);
        mma_f16(oe[vb], pa0[st], pa2[st], e0, e1);
        mma_f16(oo[vb], pa0[st], pa2[st], o0, o1);
      }
    }
  }
}

template <int G, bool kTiles, int kRing>
__device__ void run_consumer_mma_fp8(const DecodeArgs& a, int it0, int it1, const uint8_t* stages,
                                     int stage_bytes, uint64_t* full, uint64_t* empty,
                                     volatile int* abort_flag, int warp, int lane) {
  constexpr int T = kFp8Tokens;
  const int hk = warp;
  const int grp = lane >> 2;
  const int tig = lane & 3;
  const bool row_ok = grp < G;
  const uint32_t stage0 = smem_u32(stages);
  const Fp8Frags<kTiles> fr(a, hk, lane);
  bool waited = false;   // q is read at once; the first write waits (see run_consumer_mma)
  uint32_t stage = 0;
  for (int it = it0; it < it1; ++it) {
    const int32_t* item = a.sched + a.off_items + (int64_t)it * kItemWords;
    const int req = item[0], tb = item[1], te = item[2], dst = item[3];
    // q in the permuted K order: a0 = dims 16 kb + 4 tig, +1; a2 = +2, +3
    uint32_t qa0[8], qa2[8];
    float s_scale;
    {
      const uint2* qp = reinterpret_cast<const uint2*>(
          a.q + ((int64_t)req * a.hq + (int64_t)hk * G + (row_ok ? grp : 0)) * kHeadDim);
      uint2 raw[8];
      float amax = 0.f;
#pragma unroll
      for (int kb = 0; kb < 8; ++kb) {
        raw[kb] = row_ok ? __ldg(qp + kb * 4 + tig) : make_uint2(0u, 0u);
        amax = fmaxf(amax, fabsf(__uint_as_float(raw[kb].x << 16)));
        amax = fmaxf(amax, fabsf(__uint_as_float(raw[kb].x & 0xffff0000u)));
        amax = fmaxf(amax, fabsf(__uint_as_float(raw[kb].y << 16)));
        amax = fmaxf(amax, fabsf(__uint_as_float(raw[kb].y & 0xffff0000u)));
      }
      amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 2));
      const float inv = amax > 0.f ? 1.f / amax : 0.f;
#pragma unroll
      for (int kb = 0; kb < 8; ++kb) {
        qa0[kb] = pack_f16x2(__uint_as_float(raw[kb].x << 16) * inv,
                             __uint_as_float(raw[kb].x & 0xffff0000u) * inv);
        qa2[kb] = pack_f16x2(__uint_as_float(raw[kb].y << 16) * inv,
                             __uint_as_float(raw[kb].y & 0xffff0000u) * inv);
      }
      s_scale = a.scale_log2 * amax;
    }
    // accumulators per 16-dim block vb: [vb][0] even-dim tile, [vb][1] odd
    float oe[8][2], oo[8][2];
#pragma unroll
    for (int vb = 0; vb < 8; ++vb) oe[vb][0] = oe[vb][1] = oo[vb][0] = oo[vb][1] = 0.f;
    float m_run = -CUDART_INF_F;
    float l_run = 0.f;

    for (int t = tb; t < te; t += T) {
      const int n = min(T, te - t);
      const int slot = (int)(stage % kRing);
      const bool got = mbar_wait(&full[slot], (stage / kRing) & 1u, abort_flag);
      if (!__all_sync(kFull, got)) {
        if (lane == 0) raise_error(a.err, abort_flag, PKD_DEV_ERR_TIMEOUT);
        if (!waited) pdl_wait();   // complete only after the previous kernel
        return;
      }
      const uint32_t sbase = stage0 + (uint32_t)(slot * stage_bytes);
      if (n < T)
        fr.zero_v_tail(const_cast<uint8_t*>(stages) + (size_t)slot * stage_bytes, hk, lane, n);
      if (n > 16)
        fp8_stage<4, kTiles>(fr, sbase, n, tig, qa0, qa2, s_scale, oe, oo, m_run, l_run);
      else
        fp8_stage<2, kTiles>(fr, sbase, n, tig, qa0, qa2, s_scale, oe, oo, m_run, l_run);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[slot]);
      ++stage;
    }

    float l = l_run;
    l += __shfl_xor_sync(kFull, l, 1);
    l += __shfl_xor_sync(kFull, l, 2);
    if (!waited) {
      pdl_wait();
      waited = true;
    }
    if (row_ok) {
      const float inv = a.v_scale / l;
      const float lse_nat = (m_run + log2f(l)) * 0.69314718055994530942f;
      const int64_t qrow = (int64_t)req * a.hq + (int64_t)hk * G + grp;
      // lane holds dims 16 vb + 4 tig + {0, 1, 2, 3} = {oe.c0, oo.c0, oe.c1, oo.c1}
      if (dst < 0) {
        uint2* op = reinterpret_cast<uint2*>(a.out + qrow * kHeadDim) + tig;
#pragma unroll
        for (int vb = 0; vb < 8; ++vb)
          op[vb * 4] = make_uint2(pack_bf16x2(oe[vb][0] * inv, oo[vb][0] * inv),
                                  pack_bf16x2(oe[vb][1] * inv, oo[vb][1] * inv));
        if (a.lse != nullptr && tig == 0) a.lse[qrow] = lse_nat;
      } else {
        const int64_t prow = (int64_t)dst * a.hq + (int64_t)hk * G + grp;
        float4* op = reinterpret_cast<float4*>(a.o_part + prow * kHeadDim) + tig;
#pragma unroll
        for (int vb = 0; vb < 8; ++vb)
          op[vb * 4] = make_float4(oe[vb][0] * inv, oo[vb][0] * inv, oe[vb][1] * inv,
                                   oo[vb][1] * inv);
        if (tig == 0) a.l_part[prow] = lse_nat;
      }
    }
  }
}

// Stage bytes: token rows keep a padded row stride; page tiles are dense
// (16 * row_bytes per box, a multiple of 1024, so every box stays aligned for
// the 128-byte swizzle).
__host__ __device__ __forceinline__ int stage_bytes_for(int row_bytes, int tokens, bool tiles) {
  return 2 * tokens * (tiles ? row_bytes : row_stride(row_bytes));
}

// The decode role over the dynamic shared memory at `smem`: the whole
// decode kernel, and the suffix CTAs of the cascade kernel.  Warps past the
// producer (a fused launch may have more) do nothing.
template <int G, bool kMma, bool kBlock, bool kFp8, bool kTiles, int kRingSel = 0>
__device__ __forceinline__ void decode_body(const DecodeArgs& a, uint8_t* smem) {
  constexpr int kStageTokens = kFp8 ? kFp8Tokens : kTS;
  constexpr int kRing = kRingSel > 0 ? kRingSel : ring_depth(kMma, kBlock, kFp8);
  const int stage_bytes = stage_bytes_for(a.row_bytes, kStageTokens, kTiles);
  // the 128-byte swizzle repeats every 1024 bytes: page-tile stages start on
  // a 1024-byte boundary (the launch reserves the slack)
  uint8_t* stages = smem;
  if constexpr (kTiles) stages += (1024u - (smem_u32(smem) & 1023u)) & 1023u;
  float* pbuf_all = reinterpret_cast<float*>(stages + (size_t)kRing * stage_bytes);
  float* sbuf_all = pbuf_all + kMaxKvHeads * kTS * G;
  uint64_t* full = reinterpret_cast<uint64_t*>(sbuf_all + kMaxKvHeads * 32);
  uint64_t* empty = full + kRing;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kRing);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_cons = a.hkv;
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < kRing; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], (uint32_t)n_cons);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // Programmatic dependent launch: this grid may start while the previous
  // kernel in the stream still runs.  The schedule is only ever written by
  // host-to-device copies, which order fully before this kernel, and the KV
  // cache is never written by a kernel that lets its dependents start early
  // (the merge and prefix kernels do not write it; the append kernel and any
  // kernel launched without the programmatic attribute release dependents
  // only when they complete), so the producer streams KV tiles at once; the
  // same holds for q, which the tensor-core consumers read at once too.  The
  // outputs and the partial states may still be read by the previous kernel
  // (the merge of the previous layer reads the partial-state slots): every
  // consumer waits (griddepcontrol.wait) before its first write, and every
  // role waits before the grid completes.
  const int it0 = a.sched[a.off_cta + blockIdx.x];
  const int it1 = a.sched[a.off_cta + blockIdx.x + 1];
  if (it0 >= it1) {
    // no work, but still complete only after the previous kernel does, so
    // that "this grid finished" keeps implying "every earlier grid finished"
    pdl_wait();
    return;
  }
  if (warp == n_cons) {
    run_producer<kStageTokens, kTiles, kRing>(a, it0, it1, stages, stage_bytes, full, empty, abort_flag,
                                       lane);
  } else if (warp < n_cons) {
    if constexpr (kFp8) {
      run_consumer_mma_fp8<G, kTiles, kRing>(a, it0, it1, stages, stage_bytes, full, empty, abort_flag,
                                      warp, lane);
    } else if constexpr (kBlock) {
      run_consumer_mma_block<G, kTiles, kRing>(a, it0, it1, stages, stage_bytes, full, empty,
                                        abort_flag, warp, lane);
    } else if constexpr (kMma) {
      run_consumer_mma<G, kTiles, kRing>(a, it0, it1, stages, stage_bytes, full, empty, abort_flag, warp,
                                  lane);
    } else {
      run_consumer_fma<G, kRing>(a, it0, it1, stages, stage_bytes, full, empty, abort_flag,
                          pbuf_all + warp * kTS * G, sbuf_all + warp * 32, warp, lane);
    }
  }
}

template <int G, bool kMma, bool kBlock, bool kFp8, bool kTiles>
__global__ void __launch_bounds__((kMaxKvHeads + 1) * 32, 1)
    decode_kernel(const __grid_constant__ DecodeArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  if (!schedule_ready(a.sched + H_EPOCH, a.wait_epoch, a.err)) return;
  decode_body<G, kMma, kBlock, kFp8, kTiles>(a, smem);
}

// Cascade kernel (plans made by pkd_plan_cascade): CTAs [0, n_pre) run the
// shared-prefix level's items with the dense tensor-core role, the others
// the suffix level's items with the decode role (tensor-core consumer, page
// tiles), side by side in one launch; both write partial states only.  The
// split n_pre is read from the schedule header, so a captured launch follows
// each new plan.  Roles keep their own shared-memory layouts inside the
// launch's (the larger of the two) and their own programmatic-launch rules.
template <int G>
__global__ void __launch_bounds__(tc::kTcThreads, 1)
    cascade_kernel(const __grid_constant__ CascadeArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];   // each role aligns its own layout
  if (!schedule_ready(a.suf.sched + H_EPOCH, a.suf.wait_epoch, a.suf.err)) return;
  if ((int)blockIdx.x < a.pre.sched[H_NPRE])
    tc::prefix_tc_body(a.pre, smem);
  else
    decode_body<G, true, false, false, true, kCascadeSuffixRing>(a.suf, smem);
}

template <int G, bool kTiles>
const void* kernel_ptr(const DecodeKind& k) {
  if (k.fp8) return reinterpret_cast<const void*>(&decode_kernel<G, true, false, true, kTiles>);
  if (k.block) return reinterpret_cast<const void*>(&decode_kernel<G, true, true, false, kTiles>);
  if (k.mma) return reinterpret_cast<const void*>(&decode_kernel<G, true, false, false, kTiles>);
  if constexpr (kTiles) return nullptr;   // the CUDA-core consumer reads token rows only
  return reinterpret_cast<const void*>(&decode_kernel<G, false, false, false, false>);
}

template <int G>
const void* kernel_ptr_g(const DecodeKind& k) {
  return k.tmap ? kernel_ptr<G, true>(k) : kernel_ptr<G, false>(k);
}

const void* cascade_ptr(int group) {
  switch (group) {
    case 1: return reinterpret_cast<const void*>(&cascade_kernel<1>);
    case 2: return reinterpret_cast<const void*>(&cascade_kernel<2>);
    case 4: return reinterpret_cast<const void*>(&cascade_kernel<4>);
    case 8: return reinterpret_cast<const void*>(&cascade_kernel<8>);
    default: return nullptr;
  }
}

const void* kernel_for(const DecodeKind& k) {
  if (k.cascade) return (k.mma && k.tmap && !k.fp8 && !k.block) ? cascade_ptr(k.group) : nullptr;
  if (k.dense) return prefix_tc_kernel_ptr();
  if ((k.block || k.fp8) && !k.mma) return nullptr;
  if (k.block && k.fp8) return nullptr;
  switch (k.group) {
    case 1: return kernel_ptr_g<1>(k);
    case 2: return kernel_ptr_g<2>(k);
    case 4: return kernel_ptr_g<4>(k);
    case 8: return kernel_ptr_g<8>(k);
    default: return nullptr;
  }
}

}  // namespace

int decode_threads(int hkv, const DecodeKind& k) {
  if (k.cascade) return tc::kTcThreads;   // the dense role's 12 warps (the decode role uses hkv + 1)
  return k.dense ? prefix_tc_threads() : (hkv + 1) * 32;
}

bool use_mma_consumer(int group, uint32_t flags) {
  if (flags & PKD_FLAG_FMA_CONSUMER) return false;
  if (flags & PKD_FLAG_MMA_CONSUMER) return true;
  (void)group;
  return true;   // measured faster than the CUDA-core consumer at every group size
}

int decode_smem_bytes(int hkv, const DecodeKind& k) {
  if (k.dense) return prefix_tc_smem_bytes();
  const int row = hkv * kHeadDim * (k.fp8 ? 1 : 2);
  const int tokens = k.fp8 ? kFp8Tokens : kTS;
  // the cascade kernel: its decode role's ring, or the dense role's layout
  const int ring = k.cascade ? kCascadeSuffixRing : ring_depth(k.mma, k.block, k.fp8);
  const int dec = ring * stage_bytes_for(row, tokens, k.tmap) + (k.tmap ? 1024 : 0) +
                  kMaxKvHeads * kTS * k.group * 4 + kMaxKvHeads * 32 * 4 + 2 * ring * 8 + 16;
  return (k.cascade && tc::smem_bytes() > dec) ? tc::smem_bytes() : dec;
}

cudaError_t decode_prepare(const DecodeKind& k, int smem_bytes) {
  const void* f = kernel_for(k);
  if (!f) return cudaErrorInvalidValue;
  // The attribute is per kernel, shared by every context: always allow the
  // largest layout (8 KV heads) so a smaller context never lowers it.
  const int most = decode_smem_bytes(kMaxKvHeads, k);
  return cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              smem_bytes > most ? smem_bytes : most);
}

cudaError_t decode_occupancy(const DecodeKind& k, int hkv, int smem_bytes, int* blocks_per_sm) {
  const void* f = kernel_for(k);
  if (!f) return cudaErrorInvalidValue;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, f, decode_threads(hkv, k),
                                                       (size_t)smem_bytes);
}

cudaError_t launch_cascade(const DecodeKind& k, const CascadeArgs& a, int grid, int hkv,
                           int smem_bytes, cudaStream_t stream) {
  const void* f = kernel_for(k);
  if (!f || !k.cascade) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(decode_threads(hkv, k));
  cfg.dynamicSmemBytes = (size_t)smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {const_cast<CascadeArgs*>(&a)};
  return cudaLaunchKernelExC(&cfg, f, args);
}

cudaError_t launch_decode(const DecodeKind& k, const DecodeArgs& a, int grid, int hkv,
                          int smem_bytes, cudaStream_t stream) {
  const void* f = kernel_for(k);
  if (!f) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(decode_threads(hkv, k));
  cfg.dynamicSmemBytes = (size_t)smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {const_cast<DecodeArgs*>(&a)};
  return cudaLaunchKernelExC(&cfg, f, args);
}

// The map: dims (innermost first) {128-byte chunk of elements, token slot,
// 128-byte half of a head, KV head, 2 * page + (0 K, 1 V)} with byte strides
// {row, 128, D * E, P * row} (NHD) or {D * E, 128, P * D * E, P * row} (HND);
// box {chunk, 16 tokens, all halves, all heads, one K or V page}, which lands
// as [head][half][token][128 B] with the 128-byte swizzle in either layout.
namespace {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return encode;
}

}  // namespace

// The query map: dims (innermost first) {64 elements, 128-byte half, query
// head within the group, KV head, request} with byte strides {128, 256,
// g * 256, Hq * 256}; box {64, 1 half, g heads, 1 KV head, 128 / g
// requests}, which lands as 128 rows (request-major, head-minor) of 128
// bytes with the 128-byte swizzle: one half of a dense tile's A operand.
// Requests past the batch read as zeros.
cudaError_t encode_q_map(const void* q, int32_t batch, int32_t hq, int32_t hkv,
                         CUtensorMap* map) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (encode == nullptr) return cudaErrorNotSupported;
  if (q == nullptr || (uintptr_t)q % 16 != 0 || batch < 1 || hkv < 1 || hq % hkv != 0)
    return cudaErrorInvalidValue;
  const int32_t g = hq / hkv;
  if (g > 8 || kDenseRows % g != 0) return cudaErrorInvalidValue;
  const cuuint64_t row = (cuuint64_t)kHeadDim * 2;
  const cuuint64_t dims[5] = {64, 2, (cuuint64_t)g, (cuuint64_t)hkv, (cuuint64_t)batch};
  const cuuint64_t strides[4] = {128, row, (cuuint64_t)g * row, (cuuint64_t)hq * row};
  const cuuint32_t box[5] = {64, 1, (cuuint32_t)g, 1, (cuuint32_t)(kDenseRows / g)};
  const cuuint32_t elem_strides[5] = {1, 1, 1, 1, 1};
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(q), dims,
                            strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t encode_kv_map(const void* kv, int32_t num_pages, int32_t page_size, int32_t hkv,
                          bool fp8, bool hnd, bool head_half_box, CUtensorMap* map) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (encode == nullptr) return cudaErrorNotSupported;
  if (kv == nullptr || (uintptr_t)kv % 16 != 0 || page_size % 16 != 0 || num_pages < 1 ||
      hkv < 1 || hkv > kMaxKvHeads)
    return cudaErrorInvalidValue;
  const int E = fp8 ? 1 : 2;
  const cuuint64_t row = (cuuint64_t)hkv * kHeadDim * E;
  const cuuint64_t dims[5] = {(cuuint64_t)(128 / E), (cuuint64_t)page_size,
                              (cuuint64_t)(kHeadDim * E / 128), (cuuint64_t)hkv,
                              2 * (cuuint64_t)num_pages};
  const cuuint64_t head = (cuuint64_t)kHeadDim * E;
  const cuuint64_t strides[4] = {hnd ? head : row, 128, hnd ? (cuuint64_t)page_size * head : head,
                                 (cuuint64_t)page_size * row};
  const cuuint32_t box[5] = {(cuuint32_t)(128 / E), 16,
                             head_half_box ? 1u : (cuuint32_t)(kHeadDim * E / 128),
                             head_half_box ? 1u : (cuuint32_t)hkv, 1};
  const cuuint32_t elem_strides[5] = {1, 1, 1, 1, 1};
  const CUresult r = encode(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                            5, const_cast<void*>(kv), dims, strides, box, elem_strides,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace pkd
