// Internal definitions shared by the host runtime and the CUDA kernels of
// libpkd: workspace layout, schedule header words, kernel argument blocks.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include <cuda.h>   // CUtensorMap (encoded through the runtime's driver entry point)
#include <cuda_runtime_api.h>

#include "pkd.h"

namespace pkd {

constexpr int32_t kMagic = 0x31444B50;  // "PKD1"
constexpr int kHeadDim = 128;           // the decode kernel's D
constexpr int kMaxKvHeads = 8;          // one consumer warp per KV head
constexpr int kWarpTokens = 16;         // tokens per stage (each warp sees all 16)
// Shared-memory ring depth (stages of 16 tokens, 32 for E4M3) per consumer:
// with the bf16 tensor-core consumer two stages in flight per SM read HBM
// faster than three (fewer page-tile copies outstanding: measured on the
// Llama-shaped step, its HND form and the token-sparse batch); the consumers
// with more arithmetic per byte (E4M3, CUDA cores, shared-prefix row blocks)
// need the third stage to cover it.
__host__ __device__ constexpr int ring_depth(bool mma, bool block, bool fp8) {
  return (mma && !block && !fp8) ? 2 : 3;
}
constexpr int kDefaultAlpha = 32;
constexpr int kDefaultMinChunk = 256;
constexpr int kMergeThreads = 256;

// Schedule header words (first 32 int32 of the workspace; 19..31 are 0).
enum HeaderWord {
  H_MAGIC = 0, H_BATCH, H_HQ, H_HKV, H_D, H_P, H_NCTA, H_NITEMS, H_NUNITS,
  H_NSLOTS, H_CHUNK, H_ALPHA, H_NNZ, H_MAKESPAN, H_MINCHUNK, H_BLOCK,
  H_MAXCHUNKS,   // most chunks of any split request (0: nothing split)
  H_MAXBATCH,    // the capacities the word offsets were laid out for
  H_MAXPAGES,    //   (config max_batch and max_num_pages)
  H_NPRE,        // cascade plans: CTAs [0, H_NPRE) run the shared-prefix items
  H_PCHUNK,      // cascade plans: the shared-prefix level's chunk (tokens)
  H_EPOCH,       // the plan's epoch (epoch_word); the upload writes the header last
  H_WORDS = 32
};

// The plan epoch as a nonzero header word (1 .. 2^31 - 1, wrapping).
inline int32_t epoch_word(uint64_t epoch) {
  return (int32_t)((epoch - 1) % 0x7fffffffull) + 1;
}

// req (first of the block), tok_begin, tok_end, dst_slot, first page index,
// requests in the block, slot stride per request, KV head (dense-prefix
// plans: one KV head per item; otherwise 0 and the item covers all heads)
constexpr int kItemWords = 8;
constexpr int kDenseRows = 128;   // query rows of one dense-prefix tile

// Cascade plans (PKD_FLAG_CASCADE): a shared-prefix level, whose items the
// dense tensor-core role runs, and the requests' own suffix level, whose
// items the decode role runs, share one launch over disjoint CTA ranges and
// one reduction map.  The planner balances the two ranges with a cost model
// in suffix-token units: a suffix item costs alpha + tokens (every KV head of
// a token: 4 KB of K and V at Hkv 8), a prefix item (one KV head of a block
// of up to 128 query rows) costs (kCascadePrefixAlpha + tokens) *
// kCascadePrefixCost16 / 16.  Fitted to steps timed with the prefix CTA
// count forced over its whole range (in steps of Hkv), on the 8,192-token
// prefix x 32 requests step and on prefixes of 128 to 32,768 tokens x 16 or
// 64 requests with 128-token suffixes: the step time follows the slower
// role, a dense CTA taking about 8 ns per prefix token (one 128-token round
// per microsecond) after a fixed start, a decode CTA about 34 ns per
// suffix-token unit.  These constants put the chosen split on the fastest
// measured one, or within 2 % of its time, on every one of those steps.  The
// suffix chunk floor is lower than a plain plan's, since the suffix level
// gets only part of the grid.
#ifndef PKD_CASCADE_PREFIX_COST16
#define PKD_CASCADE_PREFIX_COST16 3
#endif
#ifndef PKD_CASCADE_PREFIX_ALPHA
#define PKD_CASCADE_PREFIX_ALPHA 512
#endif
#ifndef PKD_CASCADE_SUFFIX_FLOOR
#define PKD_CASCADE_SUFFIX_FLOOR 128
#endif
constexpr int64_t kCascadePrefixCost16 = PKD_CASCADE_PREFIX_COST16;
constexpr int64_t kCascadePrefixAlpha = PKD_CASCADE_PREFIX_ALPHA;
constexpr int64_t kCascadeSuffixFloor = PKD_CASCADE_SUFFIX_FLOOR;
constexpr int64_t kCascadePrefixFloor = 128;   // one round of the dense role
// The cascade kernel's decode role has the shared memory the dense role
// needs (about 227 KB), so its ring holds three 64 KB stages instead of the
// plain decode kernel's two: with part of the grid streaming the suffixes,
// each of those CTAs keeps more bytes in flight.
#ifndef PKD_CASCADE_SUFFIX_RING
#define PKD_CASCADE_SUFFIX_RING 3
#endif
constexpr int kCascadeSuffixRing = PKD_CASCADE_SUFFIX_RING;

// Fixed word offsets of the schedule arrays, all derived from capacities.
struct Layout {
  int64_t cta_indptr;    // [n_cta + 1]
  int64_t items;         // [max_items][kItemWords]
  int64_t units;         // [max_items][2]
  int64_t merge_indptr;  // [max_items + 1]
  int64_t page_list;     // [max_num_pages]
  int64_t words;         // schedule words (end of page_list)
  int64_t max_items;
  int64_t max_slots;     // partial-state slots
  // byte offsets inside the device workspace
  size_t err_byte;       // int32 device error word (never written by plan)
  size_t o_part_byte;    // fp32 [max_slots][Hq][D]
  size_t l_part_byte;    // fp32 [max_slots][Hq]
  size_t total_bytes;
};

inline int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

// Upper bound on work items of one plan: a split request of length l gives
// ceil(l / c) <= l / c + 1 chunks and every chunk candidate is at least
// ceil(L_kv / 4) with L_kv = ceil(sum l / n_cta), so sum_i ceil(l_i / c)
// <= 4 n_cta + batch.
inline int64_t max_items_for(int64_t max_batch, int64_t n_cta) {
  return max_batch + 4 * n_cta + 8;
}

// Requests per row block of a shared-prefix plan: the rows of one
// tensor-core tile per KV head over g query heads (16 for the mma.sync
// consumer, 128 for the dense-prefix kernel); 1 without grouping.
inline int32_t block_rows(const pkd_config& c) {
  const int32_t g = c.num_qo_heads / c.num_kv_heads;
  if (c.flags & PKD_FLAG_CASCADE) return kDenseRows / g;
  if (!(c.flags & PKD_FLAG_SHARED_PREFIX)) return 1;
  return ((c.flags & PKD_FLAG_DENSE_PREFIX) ? kDenseRows : 16) / g;
}

inline Layout make_layout(const pkd_config& c, int64_t n_cta) {
  Layout L{};
  L.max_items = max_items_for(c.max_batch, n_cta);
  // a shared-prefix block writes one slot per request and chunk
  L.max_slots = L.max_items * block_rows(c);
  // dense-prefix plans give every KV head of a block its own items:
  // items <= Hkv * blocks + 4 n_cta
  if (c.flags & PKD_FLAG_DENSE_PREFIX)
    L.max_items = (int64_t)c.num_kv_heads * c.max_batch + 4 * n_cta + 8;
  if (c.flags & PKD_FLAG_CASCADE) {
    // prefix items <= Hkv * blocks + 2 n_pre, suffix items <= batch + 2 n_suf
    // (chunks at least half the level's work bound); every request is a
    // unit whose slots are its prefix chunks then its suffix chunks:
    // prefix slots <= batch + 2 R n_pre / Hkv, suffix slots <= batch + 2 n_suf
    const int64_t R = block_rows(c);
    L.max_items = (int64_t)(c.num_kv_heads + 1) * c.max_batch + 2 * n_cta + 16;
    L.max_slots = 2 * (int64_t)c.max_batch + (2 * R / c.num_kv_heads + 2) * n_cta + 16;
  }
  L.cta_indptr = H_WORDS;
  L.items = align_up(L.cta_indptr + n_cta + 1, 8);
  L.units = L.items + L.max_items * kItemWords;
  L.merge_indptr = L.units + L.max_items * 2;
  L.page_list = align_up(L.merge_indptr + L.max_items + 1, 4);
  L.words = L.page_list + c.max_num_pages;
  size_t sched_bytes = (size_t)L.words * 4;
  L.err_byte = (size_t)align_up((int64_t)sched_bytes, 256);
  L.o_part_byte = L.err_byte + 256;
  L.l_part_byte = L.o_part_byte +
                  (size_t)L.max_slots * c.num_qo_heads * c.head_dim * sizeof(float);
  L.l_part_byte = (size_t)align_up((int64_t)L.l_part_byte, 256);
  L.total_bytes = L.l_part_byte + (size_t)L.max_slots * c.num_qo_heads * sizeof(float);
  L.total_bytes = (size_t)align_up((int64_t)L.total_bytes, 256);
  return L;
}

// Decode kernel arguments (by value; fixed per launch so launches can be
// captured -- the schedule itself is read from the workspace at run time).
struct DecodeArgs {
  const int32_t* sched;      // workspace base (schedule words)
  float* o_part;             // partial outputs, fp32 [slot][Hq][D]
  float* l_part;             // partial LSE, fp32 [slot][Hq] (natural log)
  int32_t* err;              // device error word
  const uint16_t* q;         // bf16 [B][Hq][D]
  const uint8_t* kv;         // NHD cache (bf16 or e4m3), bytes
  uint16_t* out;             // bf16 [B][Hq][D]
  float* lse;                // fp32 [B][Hq] or null
  int64_t page_bytes;        // 2 * P * row_bytes
  int64_t off_cta, off_items, off_pages;
  int64_t off_merge;         // merge_indptr (cascade prefix items take their slots from it)
  int32_t hq, hkv, page_size, num_pages;
  int32_t row_bytes;         // Hkv * D * element bytes: one token of one page, all heads
  float scale_log2;          // k_scale * log2(e) / sqrt(D)
  float v_scale;             // multiplies the output (1 for an unscaled cache)
  int32_t hnd;               // 1: cache is HND [pages][2][Hkv][P][D] (else NHD)
  int32_t kv_merged;         // token rows, page size 1: a token's K and V rows are adjacent
                             // in the cache and move in one copy
  // Page-tile producer only: 5-D map over the cache (128-byte chunk, token
  // slot, 128-byte half of a head, KV head, 2 * page + {0 K, 1 V}) whose
  // 16-token box lands in shared memory with the 128-byte swizzle.
  CUtensorMap kv_map;
  // Dense-prefix kernel only: q [B][Hq][D] as 5-D {64 dims, half, head in
  // group, KV head, request}; its box is one KV head's 128 query rows of a
  // block (128 / g requests x g heads) and one 128-byte half.
  CUtensorMap q_map;
  // Nonzero: before reading the schedule, wait (bounded) until its header
  // holds this epoch word -- the plan was uploaded on another stream with no
  // event ordering it before this launch.  0: the stream orders it.
  int32_t wait_epoch = 0;
};

// The cascade kernel's arguments: the shared-prefix role's (dense tile maps)
// and the suffix role's (all-heads page-tile map), over one schedule.
struct CascadeArgs {
  DecodeArgs pre;
  DecodeArgs suf;
};

struct MergeArgs {
  const int32_t* sched;
  const float* o_part;
  const float* l_part;
  uint16_t* out;
  float* lse;
  int64_t off_units, off_merge;
  int32_t hq;
  int32_t wait_epoch = 0;   // nonzero: read the schedule only after the decode grid completes
};

// Kernel launchers (decode_kernel.cu / merge_kernels.cu).
// Which decode kernel runs.
struct DecodeKind {
  int group = 1;       // query heads per KV head (1, 2, 4, 8)
  bool mma = true;     // tensor-core consumer (false: CUDA-core FMA)
  bool block = false;  // shared-prefix variant (work items over row blocks of requests)
  bool fp8 = false;    // the cache holds e4m3 (tensor-core consumer only)
  bool tmap = false;   // page-tile producer: one tensor-map copy per 16 tokens of K or V
                       // (P % 16 == 0, tensor-core consumers); else one copy per token row
  bool dense = false;  // dense shared-prefix kernel (tcgen05, one KV head per item)
  bool cascade = false;  // cascade kernel: dense prefix role + decode role (page tiles)
};
int decode_smem_bytes(int hkv, const DecodeKind& k);
int decode_threads(int hkv, const DecodeKind& k);
// The dense shared-prefix kernel (prefix_tc_kernel.cu).
const void* prefix_tc_kernel_ptr();
int prefix_tc_smem_bytes();
int prefix_tc_threads();
cudaError_t decode_prepare(const DecodeKind& k, int smem_bytes);
cudaError_t decode_occupancy(const DecodeKind& k, int hkv, int smem_bytes, int* blocks_per_sm);
cudaError_t launch_decode(const DecodeKind& k, const DecodeArgs& a, int grid, int hkv,
                          int smem_bytes, cudaStream_t stream);
cudaError_t launch_cascade(const DecodeKind& k, const CascadeArgs& a, int grid, int hkv,
                           int smem_bytes, cudaStream_t stream);
// Encode the page-tile map of a cache at `kv` (16-byte aligned) into `map`.
// A box is 16 tokens of all KV heads (the decode kernel) or, with
// head_half_box, 16 tokens of one 128-byte half of one KV head (the dense
// kernel, which lays the halves of 64 tokens out as two 8 KB matrices).
cudaError_t encode_kv_map(const void* kv, int32_t num_pages, int32_t page_size, int32_t hkv,
                          bool fp8, bool hnd, bool head_half_box, CUtensorMap* map);
// Encode the dense kernel's query map of q [batch][Hq][D] bf16.
cudaError_t encode_q_map(const void* q, int32_t batch, int32_t hq, int32_t hkv,
                         CUtensorMap* map);
// Consumer variant for a group size: tensor cores (mma.sync) or CUDA cores.
bool use_mma_consumer(int group, uint32_t flags);
// Merge grid for a persistent decode grid of n_cta CTAs.
inline int merge_grid_for(int n_cta) { return 8 * n_cta; }
// max_chunks: the most chunks of any split request of the plan (header word
// H_MAXCHUNKS); above kLongUnit the merge keeps several slots' loads in flight
// per warp.  Any value gives the same results.
constexpr int32_t kLongUnit = 64;
// batch_short (cascade plans: every request a unit of a few slots): units of
// at most 32 slots load all their slots in one batch per warp (4 each).
cudaError_t launch_merge_partials(const MergeArgs& a, int grid, int32_t max_chunks,
                                  cudaStream_t stream, bool batch_short = false);
cudaError_t launch_merge_states(const void* v_a, const float* s_a, const void* v_b,
                                const float* s_b, void* v_out, float* s_out,
                                int64_t rows, int head_dim, cudaStream_t stream);

cudaError_t launch_append(const void* k_new, const void* v_new, const int32_t* batch_indices,
                          const int32_t* positions, int32_t n, const int32_t* indptr,
                          const int32_t* indices, const int32_t* last_page_len, int32_t batch,
                          void* kv, int32_t num_pages, int32_t page_size, int32_t hkv,
                          int32_t head_bytes, bool hnd, int32_t* err, cudaStream_t stream);

// Host planner (planner.cpp).  Writes the schedule words into `words`.
int plan_schedule(const pkd_config& cfg, int32_t n_cta, const Layout& L,
                  const int32_t* indptr, const int32_t* indices,
                  const int32_t* last, int32_t batch, int32_t* words,
                  pkd_plan_info* info);
// Same over groups of requests sharing one table row each (group_indptr over
// requests, n_rows groups); group_indptr == nullptr gives plan_schedule.
int plan_schedule_grouped(const pkd_config& cfg, int32_t n_cta, const Layout& L,
                          const int32_t* group_indptr, int32_t n_rows, const int32_t* indptr,
                          const int32_t* indices, const int32_t* last, int32_t* words,
                          pkd_plan_info* info);
// Which format a shared-prefix step should take (pkd_advise_format).
int advise_format(const pkd_config& cfg, int32_t n_cta, const int32_t* group_indptr,
                  int32_t n_groups, const int32_t* p_indptr, const int32_t* p_last,
                  const int32_t* s_indptr, const int32_t* s_last, pkd_format_advice* out);
// A cascade plan: groups of requests (group_indptr) sharing prefix table rows
// (p_*, one row per group) and every request's own suffix table row (s_*,
// one row per request).
int plan_schedule_cascade(const pkd_config& cfg, int32_t n_cta, const Layout& L,
                          const int32_t* group_indptr, int32_t n_groups,
                          const int32_t* p_indptr, const int32_t* p_indices,
                          const int32_t* p_last, const int32_t* s_indptr,
                          const int32_t* s_indices, const int32_t* s_last, int32_t* words,
                          pkd_plan_info* info);

}  // namespace pkd
