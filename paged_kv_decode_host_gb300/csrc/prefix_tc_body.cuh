// Device code of the dense shared-prefix role (tcgen05 tensor cores, tensor
// memory), included by the translation units that launch it: the standalone
// dense-prefix kernel and the cascade kernel, whose first CTAs run it.
//
// What it computes is the decode kernel's (the attention state of every query
// row over an item's token range, FlashInfer 完全拆解, 从推理形状出发 and 在线
// Softmax 为什么允许任意切块), for plans whose items cover one KV head of a
// block of up to 128 / g requests that share a prefix (Composable Format:
// the shared prefix as an (R, 1) block).  Those requests' g query heads of
// the KV head are 128 rows of one dense tile, so the item is a real
// contraction: S = Q K^T (128 x 16 per page tile) and O += P V (128 x 128).
//
// GB300 design (one CTA per SM, 12 warps):
//  * warp 8 (producer) loads the item's Q tile once (two TMA tensor copies,
//    128 rows x 128 dims, 128-byte swizzle) and streams the KV head's K page
//    tiles into a 3-deep ring of 128-token slots; warp 10 streams V into a
//    ring of its own, so a K slot is refilled as soon as its score MMAs are
//    done instead of waiting for the round's P.V.  One TMA tensor copy moves
//    16 tokens of one 128-byte half of the head (2 KB), placed so that each
//    half of a slot is one [128 tokens][128 B] swizzled matrix -- a whole
//    round is one MMA operand however the pages are scattered;
//  * warp 9 (one lane) issues the score MMAs: per round of 128 tokens, S
//    into a double-buffered tensor-memory tile (M 128, N 128, K 128 in 8
//    steps, both operands K-major from shared memory; 128-token rounds
//    because these single-CTA MMAs run at about 2.8 k flop per cycle per SM
//    with N 64 but 5.1 k with N 128);
//  * warp 11 (one lane) issues the P.V MMAs once the softmax warps have
//    written P: O += P V (M 128, N 128, K 16 per page tile, A = P from
//    tensor memory, B = V N-major from shared memory).  Two issuing warps
//    because an issuing thread stalls while the tensor core works through
//    what it was given before: with one thread for both streams, each held
//    the other up.  Completion goes to mbarriers through tcgen05.commit,
//    which tracks the issuing thread's own MMAs;
//  * warps 0-7 (softmax; a thread holds one query row = one tensor-memory
//    lane; warps w and w + 4 share the lanes of quadrant w % 4, w taking
//    score columns 0-63 and w + 4 columns 64-127) read S with tcgen05.ld,
//    combine the pair's row maxima through tensor memory (each writes its
//    own into its first, already read, score column, a two-arrival barrier
//    per quadrant orders the exchange), keep the running max and their half
//    of the row sum in registers, write their half of P (bf16) with
//    tcgen05.st, and in the epilogue exchange the row sums the same way,
//    then read their half of O, normalise and write out / lse or the partial
//    state.  Two warps per quadrant because one warp's serial work per round
//    (128 maxima, exponentials and packs per row) took longer than the
//    round's MMAs: measured 1.12 us of a 1.44 us round at 32,768 x 64 with
//    one warp, the MMAs needing about 0.76 us; with two, 0.70 us of a
//    0.96-1.02 us round.  The max used in
//    the exponentials is only raised when a round's max exceeds it by more
//    than 2^8 (then O is rescaled in tensor memory), so most rounds touch O
//    not at all; the result is the same softmax, P stays <= 256.
// Tensor memory (512 columns): O [0, 128), S [128, 384) as two 128-column
// buffers, P [384, 512) as two 64-column buffers (16-bit pairs).
// Every wait is bounded; on timeout the kernel sets the device error word,
// stops, waits (bounded) for its copies and MMAs, frees tensor memory and
// returns.
#pragma once

#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "pkd_internal.h"
#include "sm103_ptx.cuh"

namespace pkd {
namespace tc {
namespace {

using namespace dev;

// 8 softmax warps (two per tensor-memory lane quadrant), K producer,
// score-MMA warp, V producer, P.V-MMA warp
constexpr int kSoftmaxWarps = 8;
constexpr int kWarpK = 8, kWarpS = 9, kWarpV = 10, kWarpPV = 11;
constexpr int kTcThreads = 12 * 32;
constexpr int kTcStages = 3;
constexpr int kRoundTok = 128;        // tokens per round = 8 page tiles of 16
constexpr int kRoundTiles = kRoundTok / 16;
constexpr int kBoxBytes = 2048;       // 16 tokens x one 128-byte half of a KV head
constexpr int kHalfBytes = kRoundTiles * kBoxBytes;   // one half of a round: [128 tokens][128 B]
constexpr int kKvBytes = 2 * kHalfBytes;          // K (or V) of a round: two halves
constexpr int kStageBytes = 2 * kKvBytes;         // K, then V
constexpr int kQBytes = kDenseRows * kHeadDim * 2;  // 32 KB
constexpr uint32_t kTmemCols = 512;
// O [0, 128); S: two 128-column fp32 buffers [128, 384); P: two 64-column
// buffers of bf16 pairs [384, 512)
constexpr uint32_t kColO = 0, kColS = 128, kColP = 384;
constexpr uint32_t kSCols = kRoundTok, kPCols = kRoundTok / 2;
static_assert(kColP + 2 * kPCols <= kTmemCols, "tensor-memory columns");
constexpr float kRescaleLog2 = 8.f;   // raise the exponent base past 2^8 growth only

struct TcSmem {
  uint64_t fullk[kTcStages], emptyk[kTcStages];   // K ring: landed / read by the score MMAs
  uint64_t fullv[kTcStages], emptyv[kTcStages];   // V ring: landed / read by the P.V MMAs
  uint64_t qfull, qfree;
  uint64_t sfull[2], sfree[2];
  uint64_t pfull[2], pfree[2];
  uint64_t ofree, fin;
  uint64_t xch[4];   // per lane quadrant: the two softmax warps' exchanges
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(1024 + kQBytes + kTcStages * kStageBytes + sizeof(TcSmem) <= 227 * 1024,
              "dynamic shared memory of one CTA");
// dynamic shared memory of the role (with the slack for 1024-byte alignment)
constexpr int smem_bytes() { return 1024 + kQBytes + kTcStages * kStageBytes + (int)sizeof(TcSmem); }

__device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                        int32_t* err, int lane) {
  const bool ok = mbar_wait(bar, parity, abort_flag);
  if (!__all_sync(kFull, ok)) {
    if (lane == 0) raise_error(err, abort_flag, PKD_DEV_ERR_TIMEOUT);
    return false;
  }
  return true;
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor: start address, leading / stride byte
// offsets (16-byte units), descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFF) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, A
// K-major, B K-major (b_mn = 0) or N-major (1), N / 8 and M / 16.
__device__ __forceinline__ uint32_t mma_idesc(int m, int n, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)b_mn << 16) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                       bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate ? 1 : 0)
      : "memory");
}

__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                       uint32_t idesc, bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate ? 1 : 0)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// 32 columns of this warp's 32 lanes (one row per thread), 32-bit each
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st1(uint32_t taddr, uint32_t v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t tmem_ld1(uint32_t taddr) {
  uint32_t v;
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(v) : "r"(taddr) : "memory");
  return v;
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 2^x, one SFU instruction (softmax weights: relative error far below the
// bf16 rounding P gets next; -inf gives 0)
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// two floats to a bf16 pair, round to nearest even (lo in the low half)
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ int rounds_of(int tb, int te) { return (te - tb + kRoundTok - 1) / kRoundTok; }

__device__ __forceinline__ void prefix_tc_body(const DecodeArgs& a, uint8_t* smem_raw) {
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sQ = smem;
  uint8_t* stages = smem + kQBytes;
  TcSmem* sh = reinterpret_cast<TcSmem*>(stages + kTcStages * kStageBytes);
  volatile int* abort_flag = &sh->abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_launch_dependents();
  const int it0 = a.sched[a.off_cta + blockIdx.x];
  const int it1 = a.sched[a.off_cta + blockIdx.x + 1];
  if (it0 >= it1) {
    pdl_wait();
    return;
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(&sh->fullk[s], 1);
      mbar_init(&sh->emptyk[s], 1);
      mbar_init(&sh->fullv[s], 1);
      mbar_init(&sh->emptyv[s], 1);
    }
    mbar_init(&sh->qfull, 1);
    mbar_init(&sh->qfree, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&sh->sfull[b], 1);
      mbar_init(&sh->sfree[b], kSoftmaxWarps);
      mbar_init(&sh->pfull[b], kSoftmaxWarps);
      mbar_init(&sh->pfree[b], 1);
    }
    mbar_init(&sh->ofree, kSoftmaxWarps);
    for (int q = 0; q < 4; ++q) mbar_init(&sh->xch[q], 2);
    mbar_init(&sh->fin, 2);
    sh->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&sh->tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sh->tmem_base;
  const int P = a.page_size;
  const int g = a.hq / a.hkv;

  if (warp == kWarpK || warp == kWarpV) {
    // ----------------------------------------------------------- producers
    // warp 8: the Q tiles and the K ring; warp 10: the V ring.  The rings are
    // apart so that a K slot is refilled as soon as its score MMAs are done,
    // not only once the round's P.V MMAs have read its V.
    const int c = warp == kWarpK ? 0 : 1;
    uint64_t* full = c ? sh->fullv : sh->fullk;
    uint64_t* empty = c ? sh->emptyv : sh->emptyk;
    uint8_t* ring = stages + (size_t)c * kTcStages * kKvBytes;
    const uint64_t policy = l2_evict_first_policy();
    pdl_wait();   // q and the cache may come from the previous kernel
    int st = 0, nq = 0;
    bool ok = true;
    for (int it = it0; it < it1 && ok; ++it) {
      const int32_t* item = a.sched + a.off_items + (int64_t)it * kItemWords;
      const int req = item[0], tb = item[1], te = item[2], poff = item[4], head = item[7];
      // Q tile of the item (the previous item's score MMAs must be done)
      if (c == 0 && it > it0 &&
          !tc_wait(&sh->qfree, (uint32_t)((it - it0 - 1) & 1), abort_flag, a.err, lane)) {
        ok = false;
        break;
      }
      if (c == 0 && lane == 0) {
        ++nq;
        mbar_arrive_expect_tx(&sh->qfull, (uint32_t)kQBytes);
        for (int h = 0; h < 2; ++h)
          tensor_copy_g2s(sQ + h * (kQBytes / 2), &a.q_map, 0, h, 0, head, req, &sh->qfull, policy);
      }
      __syncwarp();
      // page ids of the item's 16-token tiles, 32 tiles at a time: lane i
      // holds tile base + i (tb is page-aligned, so tile i starts 16 i tokens
      // into the item's pages)
      const int ntiles = (te - tb + 15) >> 4;
      int base = -32, my_page = 0;
      for (int t = tb, k = 0; t < te; t += kRoundTok, ++st, ++k) {
        const int n = min(kRoundTok, te - t);
        const int nbox = (n + 15) >> 4;
        const int tile0 = kRoundTiles * k;
        if (tile0 + kRoundTiles > base + 32) {
          base = tile0;
          my_page = 0;
          if (base + lane < ntiles) {
            my_page = a.sched[a.off_pages + poff + (16 * (base + lane)) / P];
            if ((unsigned)my_page >= (unsigned)a.num_pages) {
              atomicOr(a.err, PKD_DEV_ERR_BOUNDS);
              my_page = 0;
            }
          }
        }
        const int slot = st % kTcStages;
        const uint32_t round = (uint32_t)(st / kTcStages);
        if (round > 0 && !tc_wait(&empty[slot], (round - 1) & 1u, abort_flag, a.err, lane)) {
          ok = false;
          break;
        }
        // lane 2 j + h (lanes 0-15) copies half h of tile j of K (c = 0) or
        // V (c = 1)
        const int j = lane >> 1, h = lane & 1;
        const int page = __shfl_sync(kFull, my_page, (tile0 + (j & 7) - base) & 31);
        if (lane == 0) mbar_arrive_expect_tx(&full[slot], (uint32_t)(2 * nbox * kBoxBytes));
        __syncwarp();
        if (j < nbox)
          tensor_copy_g2s(ring + (size_t)slot * kKvBytes + h * kHalfBytes + j * kBoxBytes,
                          &a.kv_map, 0, (t + 16 * j) % P, h, head, 2 * page + c, &full[slot],
                          policy);
      }
    }
    // drain: the last phase of every slot, and the last Q tile
    if (lane == 0) {
      for (int s = 0; s < kTcStages; ++s)
        if (st > s && !mbar_wait(&full[s], (uint32_t)(((st - 1 - s) / kTcStages) & 1), nullptr))
          atomicOr(a.err, PKD_DEV_ERR_TIMEOUT);
      if (nq > 0 && !mbar_wait(&sh->qfull, (uint32_t)((nq - 1) & 1), nullptr))
        atomicOr(a.err, PKD_DEV_ERR_TIMEOUT);
    }
  } else if (warp == kWarpS) {
    // ----------------------------------------- score MMAs (lane 0 issues)
    // S of round r: its K tiles landed, Q loaded (first round of an item)
    // and its S buffer read by the softmax warps (round r - 2).  The P.V
    // MMAs come from warp 11, so neither stream waits behind the other's
    // issue (an issuing thread stalls while the tensor core works through
    // what it was given before).
    const uint32_t q0 = smem_u32(sQ), st0 = smem_u32(stages);
    int r = 0;
    bool ok = true;
    for (int it = it0; it < it1 && ok; ++it) {
      const int32_t* item = a.sched + a.off_items + (int64_t)it * kItemWords;
      const int tb = item[1], te = item[2];
      const int nr = rounds_of(tb, te);
      if (!tc_wait(&sh->qfull, (uint32_t)((it - it0) & 1), abort_flag, a.err, lane)) {
        ok = false;
        break;
      }
      for (int k = 0; k < nr; ++k, ++r) {
        const int slot = r % kTcStages, b = r & 1;
        if (!tc_wait(&sh->fullk[slot], (uint32_t)((r / kTcStages) & 1), abort_flag, a.err, lane) ||
            (r >= 2 &&
             !tc_wait(&sh->sfree[b], (uint32_t)(((r >> 1) - 1) & 1), abort_flag, a.err, lane))) {
          ok = false;
          break;
        }
        const int n = min(kRoundTok, te - (tb + k * kRoundTok));
        if (lane == 0) {
          tc_fence_after();
          // N = the round's tokens rounded up to whole tiles (tiles past
          // them were not copied)
          const uint32_t idesc_s = mma_idesc(kDenseRows, 16 * ((n + 15) >> 4), 0);
          const uint32_t kbase = st0 + (uint32_t)(slot * kKvBytes);
          for (int kk = 0; kk < 8; ++kk)
            mma_ss(tmem + kColS + kSCols * b,
                   smem_desc(q0 + (kk >> 2) * (kQBytes / 2) + (kk & 3) * 32, 16, 1024),
                   smem_desc(kbase + (kk >> 2) * kHalfBytes + (kk & 3) * 32, 16, 1024),
                   idesc_s, kk > 0);
          mma_commit(&sh->sfull[b]);
          mma_commit(&sh->emptyk[slot]);
          if (k == nr - 1) mma_commit(&sh->qfree);   // the item's last score MMA
        }
        __syncwarp();
      }
    }
    if (lane == 0) {
      mma_commit(&sh->fin);
      if (!mbar_wait(&sh->fin, 0, nullptr)) atomicOr(a.err, PKD_DEV_ERR_TIMEOUT);
    }
    __syncwarp();
  } else if (warp == kWarpPV) {
    // ------------------------------------------ P.V MMAs (lane 0 issues)
    // P.V of round r: P written, its V tiles landed and, first round of an
    // item, the previous item's O read by the epilogue
    const uint32_t idesc_o = mma_idesc(kDenseRows, kHeadDim, 1);
    int r = 0;
    bool ok = true;
    for (int it = it0; it < it1 && ok; ++it) {
      const int32_t* item = a.sched + a.off_items + (int64_t)it * kItemWords;
      const int tb = item[1], te = item[2];
      const int nr = rounds_of(tb, te);
      for (int k = 0; k < nr; ++k, ++r) {
        const int slot = r % kTcStages, b = r & 1;
        if (!tc_wait(&sh->pfull[b], (uint32_t)((r >> 1) & 1), abort_flag, a.err, lane) ||
            !tc_wait(&sh->fullv[slot], (uint32_t)((r / kTcStages) & 1), abort_flag, a.err, lane) ||
            (k == 0 && it > it0 &&
             !tc_wait(&sh->ofree, (uint32_t)((it - it0 - 1) & 1), abort_flag, a.err, lane))) {
          ok = false;
          break;
        }
        const int n = min(kRoundTok, te - (tb + k * kRoundTok));
        const int nbox = (n + 15) >> 4;
        uint8_t* vbase = stages + (size_t)(kTcStages + slot) * kKvBytes;
        if (n & 15) {
          // slots past the item's end in the last tile: P is 0 there, but
          // 0 x NaN would poison O, so zero those V rows (both halves)
          const int v0 = n & 15;
          uint8_t* tile = vbase + (nbox - 1) * kBoxBytes;
          for (int i = lane; i < 2 * (16 - v0) * 8; i += 32) {
            const int h = i / ((16 - v0) * 8), rem = i % ((16 - v0) * 8);
            const int row = v0 + rem / 8, chunk = rem % 8;
            *reinterpret_cast<uint4*>(tile + h * kHalfBytes + row * 128 + chunk * 16) =
                make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
          __syncwarp();
        }
        if (lane == 0) {
          tc_fence_after();
          const uint32_t vb = smem_u32(vbase);
          for (int j = 0; j < nbox; ++j)
            mma_ts(tmem + kColO, tmem + kColP + kPCols * b + 8 * j,
                   smem_desc(vb + j * kBoxBytes, kHalfBytes, 1024), idesc_o, k > 0 || j > 0);
          mma_commit(&sh->pfree[b]);
          mma_commit(&sh->emptyv[slot]);
        }
        __syncwarp();
      }
    }
    if (lane == 0) {
      mma_commit(&sh->fin);
      if (!mbar_wait(&sh->fin, 0, nullptr)) atomicOr(a.err, PKD_DEV_ERR_TIMEOUT);
    }
    __syncwarp();
  } else if (warp < kSoftmaxWarps) {
    // ------------------------------------------------- softmax + epilogue
    const int quad = warp & 3, half = warp >> 2;   // lane quadrant, score / O columns half
    const int row = quad * 32 + lane;               // tile row = tensor-memory lane
    const uint32_t tq = tmem + ((uint32_t)(quad * 32) << 16);   // this quadrant's lanes
    pdl_wait();   // outputs may belong to the previous kernel
    int rho = 0;
    uint32_t xc = 0;   // exchanges with the partner warp so far (the barrier's phase)
    bool ok = true;
    // wait until the P.V MMAs of round r are done (pfree of its buffer);
    // callers keep at most one phase of lag (see the round loop)
    auto pv_wait = [&](int r) -> bool {
      if (r < 0) return true;
      return tc_wait(&sh->pfree[r & 1], (uint32_t)((r >> 1) & 1), abort_flag, a.err, lane);
    };
    // one float per row with the partner warp of this quadrant: written into
    // tensor-memory column `mine` (a column this warp has already read and
    // nothing rewrites before the partner's next exchange), the partner's
    // read from `theirs`
    auto exchange = [&](uint32_t mine, uint32_t theirs, float v, float* other) -> bool {
      tmem_st1(tq + mine, __float_as_uint(v));
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh->xch[quad]);
      if (!tc_wait(&sh->xch[quad], xc & 1u, abort_flag, a.err, lane)) return false;
      ++xc;
      tc_fence_after();
      *other = __uint_as_float(tmem_ld1(tq + theirs));
      tmem_wait_ld();
      return true;
    };
    for (int it = it0; it < it1 && ok; ++it) {
      const int32_t* item = a.sched + a.off_items + (int64_t)it * kItemWords;
      const int req = item[0], tb = item[1], te = item[2], dst = item[3];
      const int n_req = item[5], stride = item[6], head = item[7];
      const int nr = rounds_of(tb, te);
      const int r0 = rho;
      float m_used = -CUDART_INF_F, l = 0.f;   // l: this warp's half of the row sum
      bool o_has = false;
      for (int k = 0; k < nr && ok; ++k) {
        const int r = r0 + k, b = r & 1;
        const int n = min(kRoundTok, te - (tb + k * kRoundTok));
        if (!tc_wait(&sh->sfull[b], (uint32_t)((r >> 1) & 1), abort_flag, a.err, lane)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // this warp's 64 score columns
        const uint32_t s_col = kColS + kSCols * b + 64 * half;
        uint32_t sv[2][32];
        tmem_ld32(tq + s_col, sv[0]);
        tmem_ld32(tq + s_col + 32, sv[1]);
        tmem_wait_ld();
        // slots past the item's end (a partial last round, the same n for
        // every row) are -inf so that their weights come out 0
        if (n < kRoundTok) {
#pragma unroll
          for (int q = 0; q < 2; ++q)
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (64 * half + 32 * q + j >= n) sv[q][j] = __float_as_uint(-CUDART_INF_F);
        }
        float mq[4] = {-CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F};
#pragma unroll
        for (int q = 0; q < 2; ++q)
#pragma unroll
          for (int j = 0; j < 32; ++j) mq[j & 3] = fmaxf(mq[j & 3], __uint_as_float(sv[q][j]));
        const float m_half = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
        // the row max of both halves (the raw scores; the scale is positive)
        float m_other;
        if (!exchange(s_col, kColS + kSCols * b + 64 * (1 - half), m_half, &m_other)) {
          ok = false;
          break;
        }
        // both halves of S are read and exchanged: the buffer may be refilled
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh->sfree[b]);
        const float mx = fmaxf(m_half, m_other) * a.scale_log2;
        // P buffer b was read by the P.V MMAs of round r - 2
        if (r >= 2 && !pv_wait(r - 2)) {
          ok = false;
          break;
        }
        // The decision is per row and the same in both warps of the pair,
        // but the waits and the tensor-memory loads / stores below are
        // warp-collective: the whole warp takes the branch when any row
        // needs it, rows that do not keep alpha = 1.  Each warp rescales its
        // half of O.
        const bool need = mx > m_used + kRescaleLog2;
        if (__any_sync(kFull, need)) {
          const float alpha = need ? exp2f(m_used - mx) : 1.f;   // 0 while m_used = -inf
          if (o_has) {
            if (!pv_wait(r - 1)) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int cb = 0; cb < 64; cb += 32) {
              uint32_t o[32];
              tmem_ld32(tq + kColO + 64 * half + cb, o);
              tmem_wait_ld();
#pragma unroll
              for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
              tmem_st32(tq + kColO + 64 * half + cb, o);
            }
            tmem_wait_st();
          }
          l *= alpha;
          if (need) m_used = mx;
        }
        // weights 2^(s scale_log2 - m_used), one FMA and one exp2 each; P
        // column c of the buffer holds tokens 2c and 2c + 1: this warp's 64
        // tokens are its 32 columns
        float ps[4] = {0.f, 0.f, 0.f, 0.f};
        const float neg_m = -m_used;
        uint32_t pw[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const uint32_t* src = sv[j >> 4];
          const int c = 2 * (j & 15);
          const float p0 = fast_exp2(fmaf(__uint_as_float(src[c]), a.scale_log2, neg_m));
          const float p1 = fast_exp2(fmaf(__uint_as_float(src[c + 1]), a.scale_log2, neg_m));
          ps[j & 3] += p0;
          ps[(j + 2) & 3] += p1;
          pw[j] = pack_bf16(p0, p1);
        }
        tmem_st32(tq + kColP + kPCols * b + 32 * half, pw);
        l += (ps[0] + ps[1]) + (ps[2] + ps[3]);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh->pfull[b]);
        o_has = true;
      }
      if (!ok) break;
      // ---- epilogue: the item's P.V MMAs done (rounds in order; lag <= 1)
      const int rl = r0 + nr - 1;
      if (!pv_wait(rl - 1) || !pv_wait(rl)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // the row sum of both halves, exchanged through the last round's P
      // columns (read by its P.V MMAs already); added in half order
      const uint32_t p_last = kColP + kPCols * (rl & 1);
      float l_other;
      if (!exchange(p_last + 32 * half, p_last + 32 * (1 - half), l, &l_other)) {
        ok = false;
        break;
      }
      const float lt = half == 0 ? l + l_other : l_other + l;
      const int i = row / g, hq = head * g + row % g;
      const bool valid = i < n_req;
      // the row's partial-state slot: dst + i * stride, or (cascade prefix
      // items, stride -1) the request's first slot plus the chunk index dst
      const int64_t slot =
          !valid ? 0
                 : (stride >= 0 ? (int64_t)dst + (int64_t)i * stride
                                : (int64_t)a.sched[a.off_merge + req + i] + dst);
      const float inv = a.v_scale / lt;
      const float lse_nat = (m_used + log2f(lt)) * 0.69314718055994530942f;
      for (int cb = 64 * half; cb < 64 * half + 64; cb += 32) {
        uint32_t o[32];
        tmem_ld32(tq + kColO + cb, o);
        tmem_wait_ld();
        if (valid) {
          if (dst < 0) {
            uint4* op = reinterpret_cast<uint4*>(
                a.out + ((int64_t)(req + i) * a.hq + hq) * kHeadDim + cb);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
              op[q4] = make_uint4(
                  pack_bf16(__uint_as_float(o[8 * q4 + 0]) * inv, __uint_as_float(o[8 * q4 + 1]) * inv),
                  pack_bf16(__uint_as_float(o[8 * q4 + 2]) * inv, __uint_as_float(o[8 * q4 + 3]) * inv),
                  pack_bf16(__uint_as_float(o[8 * q4 + 4]) * inv, __uint_as_float(o[8 * q4 + 5]) * inv),
                  pack_bf16(__uint_as_float(o[8 * q4 + 6]) * inv, __uint_as_float(o[8 * q4 + 7]) * inv));
          } else {
            float4* op = reinterpret_cast<float4*>(a.o_part + (slot * a.hq + hq) * kHeadDim + cb);
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4)
              op[q4] = make_float4(__uint_as_float(o[4 * q4]) * inv, __uint_as_float(o[4 * q4 + 1]) * inv,
                                   __uint_as_float(o[4 * q4 + 2]) * inv,
                                   __uint_as_float(o[4 * q4 + 3]) * inv);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sh->ofree);
      if (valid && half == 0) {
        if (dst < 0) {
          if (a.lse != nullptr) a.lse[(int64_t)(req + i) * a.hq + hq] = lse_nat;
        } else {
          a.l_part[slot * a.hq + hq] = lse_nat;
        }
      }
      rho = r0 + nr;
    }
  }
  // all roles done: tensor memory is no longer read or written
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kTmemCols)
                 : "memory");
  }
}

}  // namespace
}  // namespace tc
}  // namespace pkd
