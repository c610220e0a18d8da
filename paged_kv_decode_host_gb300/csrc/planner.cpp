// Host scheduler ("inspector") for paged-KV decode.
//
// Runs once per decode step on the CPU and writes a flat int32 schedule that
// the persistent decode kernel and the merge kernel read from a fixed-address
// workspace.  Rules (FlashInfer 完全拆解, 先切长 KV，再做最长任务优先分配 and
// 固定指针比固定内容更重要; FlashInfer, in depth, "Load balancing with
// split-KV"):
//
//  * table check + lengths: l_i = P (n_i - 1) + r_i, 1 <= r_i <= P, every
//    request owns >= 1 page, page ids inside the pool;
//  * work bound L_kv = ceil(sum_i l_i / N_CTA) -- one query token per
//    request, and one work item covers all KV heads of its tokens (the GQA
//    group is folded in, and an NHD page is one contiguous block for all
//    heads);
//  * chunk = L_kv rounded up to whole pages and at least the split floor
//    (short requests are not split); candidates L_kv, L_kv/2, L_kv/4 are each
//    scheduled and the smallest predicted makespan wins (ties: larger chunk);
//    with PKD_FLAG_CHUNK_SEARCH instead the largest page-multiple chunk (not
//    below the floor) whose split still gives at least N_CTA items, found by
//    binary search (pyshine FlashInfer tour, "Planning on the Host, Executing
//    on the Device": the prefill planner's search, here applied to decode);
//  * item cost alpha + tokens; items sorted by descending cost (ties: request,
//    then chunk), each given to the least-loaded CTA (ties: lowest CTA id);
//  * reduction map: split requests get contiguous partial slots in chunk
//    order; unsplit items write straight to the output (slot -1), so no
//    atomics and a fixed merge order;
//  * page ids go to the device as the CSR indices array itself; each item
//    records the index of its first page (chunks start on page boundaries).
#include <algorithm>
#include <cstring>
#include <functional>
#include <queue>
#include <utility>
#include <vector>

#include "pkd_internal.h"

namespace pkd {
namespace {

struct Item {
  int64_t cost;
  int32_t req;
  int32_t chunk_idx;
  int32_t tok_begin;
  int32_t tok_end;
};

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Largest multiple of P, at least floor_c (itself a multiple of P), whose
// split gives >= n_cta items; floor_c when none does.  The item count only
// falls as the chunk grows, so the largest such chunk is a binary search
// over whole pages.  Up to the longest request rounded up: beyond it nothing
// splits.
int64_t search_chunk(const std::vector<int64_t>& lens, int64_t n_cta, int64_t P, int64_t floor_c) {
  int64_t max_l = 0;
  for (int64_t l : lens) max_l = std::max(max_l, l);
  auto fills = [&](int64_t pages) {
    const int64_t c = pages * P;
    int64_t n = 0;
    for (int64_t l : lens) {
      n += ceil_div(l, c);
      if (n >= n_cta) return true;
    }
    return false;
  };
  int64_t lo = floor_c / P, hi = std::max(ceil_div(max_l, P), lo);
  if (!fills(lo)) return floor_c;
  while (lo < hi) {   // fills(lo) holds
    const int64_t mid = lo + (hi - lo + 1) / 2;
    if (fills(mid))
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo * P;
}

// Copy n page ids and check 0 <= id < num_pages, in one pass the compiler
// can vectorise (no early exit).
bool copy_checked(const int32_t* __restrict__ src, int32_t* __restrict__ dst, int64_t n,
                  int32_t num_pages) {
  int32_t lo = 0, hi = 0;
  for (int64_t k = 0; k < n; ++k) {
    const int32_t v = src[k];
    dst[k] = v;
    lo = v < lo ? v : lo;
    hi = v > hi ? v : hi;
  }
  return lo >= 0 && hi < num_pages;
}

// LPT visiting order: descending cost, then request, then chunk.
bool lpt_before(const Item& x, const Item& y) {
  if (x.cost != y.cost) return x.cost > y.cost;
  if (x.req != y.req) return x.req < y.req;
  return x.chunk_idx < y.chunk_idx;
}

// Split every request into chunks and return the items already in LPT
// visiting order.  Whole chunks all cost alpha + chunk and come out of the
// split in (request, chunk) order, which is their sorted order; only the
// shorter items (one per request at most) need sorting, then one merge.
void split_sorted(const std::vector<int64_t>& lens, int64_t chunk, int64_t alpha,
                  std::vector<Item>* whole, std::vector<Item>* rest, std::vector<Item>* out) {
  whole->clear();
  rest->clear();
  size_t n = 0;
  for (int64_t l : lens) n += (size_t)ceil_div(l, chunk);
  whole->reserve(n);
  rest->reserve(lens.size());
  out->reserve(n);
  for (size_t i = 0; i < lens.size(); ++i) {
    int32_t k = 0;
    for (int64_t t = 0; t < lens[i]; t += chunk, ++k) {
      const int64_t e = std::min(t + chunk, lens[i]);
      const Item it{alpha + (e - t), (int32_t)i, k, (int32_t)t, (int32_t)e};
      (e - t == chunk ? whole : rest)->push_back(it);
    }
  }
  std::sort(rest->begin(), rest->end(), lpt_before);
  out->resize(whole->size() + rest->size());
  std::merge(whole->begin(), whole->end(), rest->begin(), rest->end(), out->begin(), lpt_before);
}

// Longest processing time first over items given in visiting order.
// Returns the makespan and the CTA of each item.  The CTA loads sit in a
// flat binary min-heap keyed by (load, CTA id); giving an item to the top
// CTA only grows its key, so one sift-down per item keeps the heap (the same
// choice as pop + push, at half the work).  The leading run of equal-cost
// items (the whole chunks) needs no heap: from equal loads, ties by CTA id
// hand them out round-robin, so item j of the run goes to CTA j mod n_cta;
// the heap is built once after it.  Keys are unique (CTA ids), so any valid
// heap gives the same choices.
void sift_down(std::pair<int64_t, int32_t>* h, size_t n, size_t i) {
  const std::pair<int64_t, int32_t> v = h[i];
  for (;;) {
    size_t c = 2 * i + 1;
    if (c >= n) break;
    if (c + 1 < n && h[c + 1] < h[c]) ++c;
    if (!(h[c] < v)) break;
    h[i] = h[c];
    i = c;
  }
  h[i] = v;
}

int64_t lpt(const std::vector<Item>& items, int32_t n_cta, std::vector<int32_t>* owner,
            std::vector<std::pair<int64_t, int32_t>>* heap) {
  heap->resize((size_t)n_cta);
  std::pair<int64_t, int32_t>* h = heap->data();
  owner->resize(items.size());
  const size_t n = (size_t)n_cta;
  // leading equal-cost run: round-robin
  size_t k = 0;
  const int64_t w0 = items.empty() ? 0 : items[0].cost;
  while (k < items.size() && items[k].cost == w0) {
    (*owner)[k] = (int32_t)(k % n);
    ++k;
  }
  const int64_t q = (int64_t)(k / n), r = (int64_t)(k % n);
  for (int32_t c = 0; c < n_cta; ++c) h[c] = std::make_pair(w0 * (q + (c < r ? 1 : 0)), c);
  int64_t makespan = w0 * (q + (r > 0 ? 1 : 0));
  if (r > 0)   // loads are not all equal: order them into a heap
    for (size_t i = n / 2; i-- > 0;) sift_down(h, n, i);
  for (size_t idx = k; idx < items.size(); ++idx) {
    (*owner)[idx] = h[0].second;
    h[0].first += items[idx].cost;
    makespan = std::max(makespan, h[0].first);
    sift_down(h, n, 0);
  }
  return makespan;
}

struct Block {
  int32_t req_first, n_req, table_row;
};

// Working arrays of one plan, kept per host thread between calls: the planner
// runs every decode step, and reusing their storage takes the allocator off
// that path.  Every array is cleared or resized before use.
struct Scratch {
  std::vector<int64_t> row_len, lens, unit_lens, cands;
  std::vector<Block> blocks;
  std::vector<Item> items, best_items, whole, rest;
  std::vector<int32_t> owner, best_owner, first_slot, n_chunks, count, fill, by_pos, split_blocks;
  std::vector<std::pair<int64_t, int32_t>> heap;
  std::vector<std::pair<int32_t, int32_t>> units;
};

}  // namespace

int plan_schedule(const pkd_config& cfg, int32_t n_cta, const Layout& L,
                  const int32_t* indptr, const int32_t* indices, const int32_t* last,
                  int32_t batch, int32_t* words, pkd_plan_info* info) {
  return plan_schedule_grouped(cfg, n_cta, L, nullptr, batch, indptr, indices, last, words,
                               info);
}

// Row blocks: a block is a run of consecutive requests that attend over the
// same pages (table row).  Without grouping every request is its own block;
// with grouping (a shared prefix, FlashInfer 完全拆解, Composable Format) the
// requests of a group are cut into blocks of `rows` requests -- the query
// rows one tensor-core tile holds per KV head (16 / g for the mma.sync
// consumer, 128 / g for the dense-prefix kernel) -- so one read of the
// group's pages serves the whole block.  Dense-prefix plans split the work
// of a block further by KV head: the unit of work is (block, head), and the
// chunk bound, the split and LPT run over those units.
int plan_schedule_grouped(const pkd_config& cfg, int32_t n_cta, const Layout& L,
                          const int32_t* group_indptr, int32_t n_rows, const int32_t* indptr,
                          const int32_t* indices, const int32_t* last, int32_t* words,
                          pkd_plan_info* info) {
  // n_rows: table rows (= requests without grouping, = groups with it)
  if (n_rows < 0 || n_cta < 1 || words == nullptr) return PKD_E_INVALID_ARG;
  if (n_rows > 0 && (indptr == nullptr || last == nullptr)) return PKD_E_INVALID_ARG;
  const int64_t P = cfg.page_size;
  const int32_t group = cfg.num_qo_heads / cfg.num_kv_heads;
  const int32_t rows = group_indptr ? block_rows(cfg) : 1;
  const int32_t heads = (group_indptr && (cfg.flags & PKD_FLAG_DENSE_PREFIX))
                            ? cfg.num_kv_heads : 1;   // units per block
  (void)group;

  // requests
  int32_t batch = n_rows;
  if (group_indptr) {
    if (group_indptr[0] != 0) return PKD_E_BAD_TABLE;
    for (int32_t j = 0; j < n_rows; ++j)
      if (group_indptr[j + 1] <= group_indptr[j]) return PKD_E_BAD_TABLE;
    batch = n_rows > 0 ? group_indptr[n_rows] : 0;
  }
  if (batch > cfg.max_batch) return PKD_E_CAPACITY;

  thread_local Scratch sc;
  // ---- P0: table check and lengths (per table row)
  std::vector<int64_t>& row_len = sc.row_len;
  row_len.resize((size_t)n_rows);
  int64_t nnz = 0;
  if (n_rows > 0) {
    if (indptr[0] != 0) return PKD_E_BAD_TABLE;
    for (int32_t i = 0; i < n_rows; ++i) {
      int64_t n = (int64_t)indptr[i + 1] - indptr[i];
      if (n < 1) return PKD_E_BAD_TABLE;
      if (last[i] < 1 || last[i] > P) return PKD_E_BAD_TABLE;
      row_len[i] = P * (n - 1) + last[i];
      if (row_len[i] > 0x7fffffffLL) return PKD_E_CAPACITY;
    }
    nnz = indptr[n_rows];
    if (nnz > cfg.max_num_pages) return PKD_E_CAPACITY;
    if (nnz > 0 && indices == nullptr) return PKD_E_INVALID_ARG;
    // page ids go into the schedule verbatim (the kernel reads a table row's
    // pages at indptr[row] + t / P), range-checked in the same pass
    if (!copy_checked(indices, words + L.page_list, nnz, cfg.num_pages)) return PKD_E_BAD_TABLE;
  }

  // ---- row blocks
  std::vector<Block>& blocks = sc.blocks;
  std::vector<int64_t>& lens = sc.lens;  // per block: tokens of its table row
  blocks.clear();
  lens.clear();
  if (group_indptr) {
    for (int32_t j = 0; j < n_rows; ++j)
      for (int32_t r = group_indptr[j]; r < group_indptr[j + 1]; r += rows) {
        blocks.push_back(Block{r, std::min(rows, group_indptr[j + 1] - r), j});
        lens.push_back(row_len[j]);
      }
  } else {
    for (int32_t i = 0; i < n_rows; ++i) blocks.push_back(Block{i, 1, i});
    lens.assign(row_len.begin(), row_len.end());
  }
  const int32_t n_blocks = (int32_t)blocks.size();
  // work units: block-major, head-minor (unit u = block u / heads, head u % heads)
  std::vector<int64_t>& unit_lens = sc.unit_lens;
  unit_lens.clear();
  if (heads > 1) {
    for (int64_t l : lens)
      for (int32_t hk = 0; hk < heads; ++hk) unit_lens.push_back(l);
  }
  const std::vector<int64_t>& ulens = heads > 1 ? unit_lens : lens;
  int64_t total = 0;
  for (int64_t l : ulens) total += l;

  // ---- P1 + P2 + P3: chunk candidates, split, LPT; keep the best
  const int64_t alpha = cfg.alpha < 0 ? kDefaultAlpha : cfg.alpha;
  const int64_t min_chunk = cfg.min_chunk_tokens < 0 ? kDefaultMinChunk : cfg.min_chunk_tokens;
  const int64_t floor_c = ceil_div(std::max<int64_t>(min_chunk, 1), P) * P;
  const int64_t work_bound = ceil_div(total, n_cta);
  std::vector<int64_t>& cands = sc.cands;
  cands.clear();
  if (cfg.flags & PKD_FLAG_CHUNK_SEARCH) {
    cands.push_back(search_chunk(ulens, n_cta, P, floor_c));
  } else {
    for (int64_t k : {1, 2, 4}) {
      int64_t c = std::max(ceil_div(ceil_div(work_bound, k), P) * P, floor_c);
      if (std::find(cands.begin(), cands.end(), c) == cands.end()) cands.push_back(c);
    }
  }
  std::vector<Item>& items = sc.items;
  std::vector<Item>& best_items = sc.best_items;
  std::vector<int32_t>& owner = sc.owner;
  std::vector<int32_t>& best_owner = sc.best_owner;
  int64_t best_chunk = -1, best_span = 0;
  for (int64_t c : cands) {
    if (best_chunk >= 0) {
      // a later (smaller) candidate must beat the best makespan strictly;
      // skip it when even its lower bound -- its costliest item, or its total
      // cost spread evenly -- cannot
      int64_t n_it = 0, top = 0;
      for (int64_t l : ulens) {
        n_it += ceil_div(l, c);
        top = std::max(top, std::min(l, c));
      }
      const int64_t lb = std::max(alpha + top, ceil_div(total + alpha * n_it, n_cta));
      if (lb >= best_span) continue;
    }
    split_sorted(ulens, c, alpha, &sc.whole, &sc.rest, &items);
    int64_t span = lpt(items, n_cta, &owner, &sc.heap);
    if (best_chunk < 0 || span < best_span) {
      best_chunk = c;
      best_span = span;
      best_items.swap(items);
      best_owner.swap(owner);
    }
  }
  const int64_t n_items = (int64_t)best_items.size();
  if (n_items > L.max_items) return PKD_E_CAPACITY;

  // ---- P4: reduction map: every request of a split block is a unit with
  // one slot per chunk, slots in chunk order.  Units go longest first (most
  // chunks; ties: ascending request), so that the merge's longest tasks are
  // handed out first when its tasks take more than one wave of blocks.
  std::vector<int32_t>& first_slot = sc.first_slot;  // slot of the block's first request
  std::vector<int32_t>& n_chunks = sc.n_chunks;
  std::vector<std::pair<int32_t, int32_t>>& units = sc.units;
  std::vector<int32_t>& split_blocks = sc.split_blocks;
  first_slot.assign((size_t)n_blocks, -1);
  n_chunks.assign((size_t)n_blocks, 1);
  units.clear();
  split_blocks.clear();
  for (int32_t b = 0; b < n_blocks; ++b) {
    n_chunks[b] = (int32_t)ceil_div(lens[b], best_chunk);
    if (n_chunks[b] > 1) split_blocks.push_back(b);
  }
  std::stable_sort(split_blocks.begin(), split_blocks.end(),
                   [&](int32_t x, int32_t y) { return n_chunks[x] > n_chunks[y]; });
  int64_t n_slots = 0;
  for (int32_t b : split_blocks) {
    const int32_t nc = n_chunks[b];
    first_slot[b] = (int32_t)n_slots;
    for (int32_t r = 0; r < blocks[b].n_req; ++r) {
      units.emplace_back(blocks[b].req_first + r, nc);
      n_slots += nc;
    }
  }
  if (n_slots > L.max_slots || (int64_t)units.size() > L.max_items) return PKD_E_CAPACITY;

  // ---- serialize: queues in CTA order, each in assignment (LPT) order
  std::vector<int32_t>& count = sc.count;
  count.assign((size_t)n_cta, 0);
  for (int64_t j = 0; j < n_items; ++j) count[best_owner[j]]++;
  int32_t* cta_indptr = words + L.cta_indptr;
  cta_indptr[0] = 0;
  for (int32_t c = 0; c < n_cta; ++c) cta_indptr[c + 1] = cta_indptr[c] + count[c];
  std::vector<int32_t>& fill = sc.fill;
  std::vector<int32_t>& by_pos = sc.by_pos;
  fill.assign(cta_indptr, cta_indptr + n_cta);
  by_pos.resize((size_t)n_items);
  for (int64_t j = 0; j < n_items; ++j) by_pos[fill[best_owner[j]]++] = (int32_t)j;

  int32_t* item_words = words + L.items;
  for (int64_t p = 0; p < n_items; ++p) {
    const Item& it = best_items[by_pos[p]];
    const int32_t b = it.req / heads;   // it.req is the unit
    const Block& bk = blocks[b];
    int32_t* w = item_words + p * kItemWords;
    w[0] = bk.req_first;
    w[1] = it.tok_begin;
    w[2] = it.tok_end;
    w[3] = first_slot[b] >= 0 ? first_slot[b] + it.chunk_idx : -1;
    w[4] = (int32_t)(indptr[bk.table_row] + it.tok_begin / P);  // index of the first page
    w[5] = bk.n_req;
    w[6] = first_slot[b] >= 0 ? n_chunks[b] : 0;     // slot stride per request
    w[7] = it.req % heads;                           // KV head (dense prefix), else 0
  }
  int32_t* unit_words = words + L.units;
  int32_t* merge_indptr = words + L.merge_indptr;
  merge_indptr[0] = 0;
  for (size_t u = 0; u < units.size(); ++u) {
    unit_words[2 * u] = units[u].first;
    unit_words[2 * u + 1] = units[u].second;
    merge_indptr[u + 1] = merge_indptr[u] + units[u].second;
  }

  int32_t* h = words;
  std::memset(h, 0, sizeof(int32_t) * H_WORDS);
  h[H_MAGIC] = kMagic;
  h[H_BATCH] = batch;
  h[H_HQ] = cfg.num_qo_heads;
  h[H_HKV] = cfg.num_kv_heads;
  h[H_D] = cfg.head_dim;
  h[H_P] = cfg.page_size;
  h[H_NCTA] = n_cta;
  h[H_NITEMS] = (int32_t)n_items;
  h[H_NUNITS] = (int32_t)units.size();
  h[H_NSLOTS] = (int32_t)n_slots;
  h[H_CHUNK] = (int32_t)best_chunk;
  h[H_ALPHA] = (int32_t)alpha;
  h[H_NNZ] = (int32_t)nnz;
  h[H_MAKESPAN] = (int32_t)std::min<int64_t>(best_span, 0x7fffffff);
  h[H_MINCHUNK] = (int32_t)floor_c;
  h[H_BLOCK] = rows;
  int32_t max_chunks = 0;
  for (const auto& un : units) max_chunks = std::max(max_chunks, un.second);
  h[H_MAXCHUNKS] = max_chunks;
  h[H_MAXBATCH] = cfg.max_batch;
  h[H_MAXPAGES] = cfg.max_num_pages;

  if (info) {
    info->batch = batch;
    info->num_ctas = n_cta;
    info->chunk_tokens = (int32_t)best_chunk;
    info->num_items = (int32_t)n_items;
    info->num_units = (int32_t)units.size();
    info->num_slots = (int32_t)n_slots;
    int64_t tokens = 0;   // sum of the blocks' lengths (not per head)
    for (int64_t l : lens) tokens += l;
    info->total_tokens = tokens;
    info->makespan = best_span;
    info->nnz = (int32_t)nnz;
    info->schedule_words = (int32_t)(L.page_list + nnz);
  }
  return PKD_OK;
}

// ---------------------------------------------------------------- cascade
//
// One decode step with a shared-prefix level and a suffix level, planned
// together ("FlashInfer, in depth", "Cascades, Merges, and the Autotuner":
// attention once per level, then a merge; "FlashInfer 完全拆解", Composable
// Format and 先切长 KV，再做最长任务优先分配).  The grid is cut in two: CTAs
// [0, n_pre) take the prefix items -- over units (block of up to R requests
// of a group, KV head) as in a dense-prefix plan -- and CTAs [n_pre, n_cta)
// the suffix items -- over units (request), all KV heads, as in a plain
// plan, with the closed-form chunk of the suffix level's own work bound (and
// its half) and LPT on its own CTAs.
//
// The prefix level gives every CTA at most one item (a dense CTA's second
// item waits for its query tile and its first item's epilogue, which costs
// more than a longer first item): with a budget of n CTAs, every block
// starts with one chunk per KV head, and while Hkv more CTAs are left the
// block whose chunk is longest (ties: the first block) gets one more chunk
// per head -- every head of a block keeps the same chunks, so a request's
// prefix slots hold all its heads -- unless that would cut it below the
// floor; then each block keeps the fewest chunks that stay within the
// longest chunk.  Chunks are page-rounded (a block may end up with fewer than its
// share); item j goes to CTA j and unused budget goes to the suffix level.
// When the blocks' heads outnumber the grid, the prefix units are not split
// and LPT places them on the n_pre CTAs instead.
//
// n_pre balances the two levels' predicted makespans in one cost unit
// (suffix tokens: kCascadePrefixCost16): starting from the budget that gives
// each level CTAs in proportion to its total cost (in steps of Hkv when
// every head can have a CTA, rounded to the nearest step), it moves toward
// its better neighbour budget (the next one either way whose prefix level
// differs), if that one is strictly better, and on from neighbour to
// neighbour while the budget keeps improving strictly.  Budgets compare by
// the predicted makespan, ties by the sum of both levels'.  Every item writes a partial state: request r's slots are
// merge_indptr[r] .. merge_indptr[r + 1], its prefix chunks first, then its
// suffix chunks, and one merge folds them.  Prefix items mark themselves with
// slot stride -1 and carry their chunk index as dst_slot (a block's requests
// have different slot bases); suffix items carry their slot.
namespace {

struct LevelPlan {
  int64_t chunk = 0, span = 0;
  std::vector<Item> items;
  std::vector<int32_t> owner;
  std::vector<int64_t> block_chunk;   // prefix level: the chunk of each block
  int32_t ctas = 0;                   // prefix level: CTAs its items use
};

// Closed-form chunk candidates (the work bound over n CTAs, and its half),
// page-rounded and not below floor_c; the smaller predicted makespan wins
// (ties: the larger chunk).  A candidate whose makespan lower bound (its
// costliest item, or its total cost spread evenly) cannot beat the best so
// far is not scheduled.
// Split results already computed for these lengths, by chunk (one search
// evaluates several budgets, and their candidates often share a chunk).
// Entries past `used` keep their storage for the next search.
struct SplitCache {
  std::vector<std::pair<int64_t, std::vector<Item>>> e;
  size_t used = 0;
};

void plan_level(const std::vector<int64_t>& ulens, int64_t total, int32_t n, int64_t P,
                int64_t floor_c, int64_t alpha, Scratch& sc, LevelPlan* out,
                SplitCache* cache = nullptr) {
  out->chunk = -1;
  const int64_t bound = ceil_div(total, n);
  int64_t prev = -1;
  for (int64_t k : {1, 2}) {
    const int64_t c = std::max(ceil_div(ceil_div(bound, k), P) * P, floor_c);
    if (c == prev) continue;
    prev = c;
    if (out->chunk >= 0) {
      int64_t n_it = 0, top = 0;
      for (int64_t l : ulens) {
        n_it += ceil_div(l, c);
        top = std::max(top, std::min(l, c));
      }
      if (std::max(alpha + top, ceil_div(total + alpha * n_it, n)) >= out->span) continue;
    }
    bool cached = false;
    if (cache != nullptr) {
      for (size_t i = 0; i < cache->used; ++i)
        if (cache->e[i].first == c) {
          sc.items.assign(cache->e[i].second.begin(), cache->e[i].second.end());
          cached = true;
          break;
        }
    }
    if (!cached) {
      split_sorted(ulens, c, alpha, &sc.whole, &sc.rest, &sc.items);
      if (cache != nullptr) {
        if (cache->used == cache->e.size()) cache->e.emplace_back();
        cache->e[cache->used].first = c;
        cache->e[cache->used].second.assign(sc.items.begin(), sc.items.end());
        ++cache->used;
      }
    }
    const int64_t span = lpt(sc.items, n, &sc.owner, &sc.heap);
    if (out->chunk < 0 || span < out->span) {
      out->chunk = c;
      out->span = span;
      out->items.swap(sc.items);
      out->owner.swap(sc.owner);
    }
  }
}

// Chunks of the prefix level on a budget of n CTAs when every (block, head)
// unit can have one (see above): water-filling, then every block keeps the
// fewest chunks whose length stays within the longest chunk (more would not
// shorten the level).  Fills m (chunks per block) and chunk; returns the
// CTAs used.
int32_t prefix_chunks(const std::vector<int64_t>& block_len, int32_t hkv, int32_t n, int64_t P,
                      int64_t floor_c, std::vector<int32_t>& m, std::vector<int64_t>& chunk) {
  const int32_t n_blocks = (int32_t)block_len.size();
  m.assign((size_t)n_blocks, 1);
  chunk.resize((size_t)n_blocks);
  for (int32_t b = 0; b < n_blocks; ++b) chunk[b] = ceil_div(block_len[b], P) * P;
  for (int64_t budget = n - (int64_t)n_blocks * hkv; budget >= hkv; budget -= hkv) {
    int32_t top = 0;
    for (int32_t b = 1; b < n_blocks; ++b)
      if (chunk[b] > chunk[top]) top = b;
    const int64_t next = ceil_div(ceil_div(block_len[top], m[top] + 1), P) * P;
    if (next < floor_c) break;
    m[top] += 1;
    chunk[top] = next;
  }
  int64_t top = 0;
  for (int64_t c : chunk) top = std::max(top, c);
  int64_t used = 0;
  for (int32_t b = 0; b < n_blocks; ++b) {
    while (m[b] > 1 && ceil_div(ceil_div(block_len[b], m[b] - 1), P) * P <= top) --m[b];
    chunk[b] = ceil_div(ceil_div(block_len[b], m[b]), P) * P;
    used += (int64_t)m[b] * hkv;
  }
  return (int32_t)used;
}

// The prefix level of a cascade plan on a budget of n CTAs (see above).
// block_len: each block's prefix length; units = blocks x hkv.
void plan_prefix(const std::vector<int64_t>& block_len, int32_t hkv, int32_t n, int64_t P,
                 int64_t floor_c, int64_t alpha, Scratch& sc, LevelPlan* out) {
  const int32_t n_blocks = (int32_t)block_len.size();
  out->items.clear();
  out->owner.clear();
  out->block_chunk.assign((size_t)n_blocks, 0);
  out->span = 0;
  if ((int64_t)n_blocks * hkv > n) {
    // unsplit (block, head) units by LPT
    sc.unit_lens.clear();
    for (int64_t l : block_len)
      for (int32_t h = 0; h < hkv; ++h) sc.unit_lens.push_back(l);
    int64_t top = 0;
    for (int64_t l : block_len) top = std::max(top, l);
    split_sorted(sc.unit_lens, std::max<int64_t>(top, 1), alpha, &sc.whole, &sc.rest,
                 &out->items);
    out->span = lpt(out->items, n, &out->owner, &sc.heap);
    for (int32_t b = 0; b < n_blocks; ++b) out->block_chunk[b] = std::max<int64_t>(top, 1);
    out->ctas = n;
    return;
  }
  prefix_chunks(block_len, hkv, n, P, floor_c, sc.n_chunks, out->block_chunk);
  for (int32_t b = 0; b < n_blocks; ++b) {
    const int64_t c = out->block_chunk[b];
    for (int32_t h = 0; h < hkv; ++h) {
      int32_t k = 0;
      for (int64_t t = 0; t < block_len[b]; t += c, ++k) {
        const int64_t e = std::min(t + c, block_len[b]);
        out->owner.push_back((int32_t)out->items.size());
        out->items.push_back(Item{alpha + (e - t), b * hkv + h, k, (int32_t)t, (int32_t)e});
        out->span = std::max(out->span, alpha + (e - t));
      }
    }
  }
  out->ctas = (int32_t)out->items.size();
}

// Table rows of one level: validate and return the lengths.
int row_lengths(const int32_t* indptr, const int32_t* last, int32_t rows, int64_t P,
                std::vector<int64_t>* len) {
  len->resize((size_t)rows);
  if (rows == 0) return PKD_OK;
  if (indptr == nullptr || last == nullptr) return PKD_E_INVALID_ARG;
  if (indptr[0] != 0) return PKD_E_BAD_TABLE;
  for (int32_t i = 0; i < rows; ++i) {
    const int64_t n = (int64_t)indptr[i + 1] - indptr[i];
    if (n < 1 || last[i] < 1 || last[i] > P) return PKD_E_BAD_TABLE;
    (*len)[i] = P * (n - 1) + last[i];
    if ((*len)[i] > 0x7fffffffLL) return PKD_E_CAPACITY;
  }
  return PKD_OK;
}

struct CascadeScratch {
  std::vector<int64_t> pre_row, suf_len, block_len;
  std::vector<Block> blocks;
  std::vector<int32_t> block_of, np_block, ns_req, count, fill;
  std::vector<int64_t> chunk_tmp;
  SplitCache split_cache;   // the suffix level's splits, by chunk, within one search
  LevelPlan pre, suf, best_pre, best_suf;
};

}  // namespace

// The cascade plan's search over the tables' lengths (no page ids): blocks,
// both levels' costs, and the CTA split; the chosen levels are left in
// cs.best_pre / cs.best_suf.  *n_pre, *span (1/16 suffix-token units) and
// *batch are set.
int cascade_search(const pkd_config& cfg, int32_t n_cta, const int32_t* group_indptr,
                   int32_t n_groups, const int32_t* p_indptr, const int32_t* p_last,
                   const int32_t* s_indptr, const int32_t* s_last, Scratch& sc, CascadeScratch& cs,
                   int32_t* batch_out, int32_t* n_pre_out, int64_t* span_out, int64_t* alpha_out,
                   int64_t* floor_s_out) {
  if (n_groups < 0 || n_cta < 2) return PKD_E_INVALID_ARG;
  if (n_groups > 0 && group_indptr == nullptr) return PKD_E_INVALID_ARG;
  const int64_t P = cfg.page_size;
  const int32_t R = block_rows(cfg);
  const int32_t hkv = cfg.num_kv_heads;
  int32_t batch = 0;
  if (n_groups > 0) {
    if (group_indptr[0] != 0) return PKD_E_BAD_TABLE;
    for (int32_t j = 0; j < n_groups; ++j)
      if (group_indptr[j + 1] <= group_indptr[j]) return PKD_E_BAD_TABLE;
    batch = group_indptr[n_groups];
  }
  if (batch > cfg.max_batch) return PKD_E_CAPACITY;
  int st = row_lengths(p_indptr, p_last, n_groups, P, &cs.pre_row);
  if (st != PKD_OK) return st;
  st = row_lengths(s_indptr, s_last, batch, P, &cs.suf_len);
  if (st != PKD_OK) return st;

  // ---- prefix blocks (units: block x KV head) and the levels' total costs
  cs.blocks.clear();
  cs.block_len.clear();
  cs.block_of.assign((size_t)batch, 0);
  int64_t pre_cost = 0;
  for (int32_t j = 0; j < n_groups; ++j)
    for (int32_t r = group_indptr[j]; r < group_indptr[j + 1]; r += R) {
      const int32_t n = std::min(R, group_indptr[j + 1] - r);
      for (int32_t i = 0; i < n; ++i) cs.block_of[r + i] = (int32_t)cs.blocks.size();
      cs.blocks.push_back(Block{r, n, j});
      cs.block_len.push_back(cs.pre_row[j]);
      pre_cost += hkv * (kCascadePrefixAlpha + cs.pre_row[j]) * kCascadePrefixCost16;
    }
  const int64_t alpha = cfg.alpha < 0 ? kDefaultAlpha : cfg.alpha;
  int64_t suf_total = 0, suf_cost = 0;
  for (int64_t l : cs.suf_len) {
    suf_total += l;
    suf_cost += (alpha + l) * 16;
  }
  const int64_t floor_s = ceil_div(
      std::max<int64_t>(cfg.min_chunk_tokens < 0 ? kCascadeSuffixFloor : cfg.min_chunk_tokens, 1),
      P) * P;
  const int64_t floor_p = ceil_div(kCascadePrefixFloor, P) * P;

  // ---- the CTA split (see above)
  int32_t n_pre = 0;
  int64_t best_span = 0;
  if (batch > 0) {
    const int64_t units = (int64_t)cs.blocks.size() * hkv;
    // budgets: units + step * j when every head can have a CTA, else 1 .. n_cta - 1
    const bool split = units <= n_cta - 1;
    const int64_t base = split ? units : 1, step = split ? hkv : 1;
    const int64_t j_max = (n_cta - 1 - base) / step;
    const int64_t all = pre_cost + suf_cost;
    const int64_t prop = (n_cta * pre_cost + all / 2) / all;
    const int64_t j0 = std::min<int64_t>(
        std::max<int64_t>((std::max<int64_t>(prop - base, 0) + step / 2) / step, 0), j_max);
    cs.split_cache.used = 0;
    int64_t best_j = -1, best_sum = 0;
    // budgets compare by the predicted makespan, ties by the sum of the two
    // levels' makespans (a budget that does not shorten the bounding level
    // but lengthens the other loses)
    auto evaluate = [&](int64_t j) {
      plan_prefix(cs.block_len, hkv, (int32_t)(base + step * j), P, floor_p, kCascadePrefixAlpha,
                  sc, &cs.pre);
      plan_level(cs.suf_len, suf_total, n_cta - cs.pre.ctas, P, floor_s, alpha, sc, &cs.suf,
                 &cs.split_cache);
      const int64_t p_span = cs.pre.span * kCascadePrefixCost16, s_span = cs.suf.span * 16;
      const int64_t span = std::max(p_span, s_span), sum = p_span + s_span;
      if (best_j < 0 || span < best_span || (span == best_span && sum < best_sum)) {
        best_span = span;
        best_sum = sum;
        best_j = j;
        std::swap(cs.best_pre, cs.pre);
        std::swap(cs.best_suf, cs.suf);
      }
    };
    // CTAs the prefix level uses at budget j, and the next budget from j in
    // direction d whose prefix level differs (budgets between give the
    // same plan), or -1
    auto used = [&](int64_t j) -> int32_t {
      const int64_t n = base + step * j;
      if (!split) return (int32_t)n;
      return prefix_chunks(cs.block_len, hkv, (int32_t)n, P, floor_p, sc.n_chunks, cs.chunk_tmp);
    };
    auto neighbour = [&](int64_t j, int64_t d) -> int64_t {
      const int32_t c = used(j);
      for (int64_t k = j + d; k >= 0 && k <= j_max; k += d)
        if (used(k) != c) return k;
      return -1;
    };
    evaluate(j0);
    // the better neighbour (the lower one on a tie), if it beats j0
    // strictly, gives the direction; then on from neighbour to neighbour
    // while the budget keeps improving strictly
    const int64_t lo = neighbour(j0, -1), hi = neighbour(j0, 1);
    if (lo >= 0) evaluate(lo);
    if (hi >= 0) evaluate(hi);
    const int64_t dir = best_j > j0 ? 1 : (best_j < j0 ? -1 : 0);
    for (int64_t j = dir != 0 ? neighbour(best_j, dir) : -1; j >= 0; j = neighbour(j, dir)) {
      evaluate(j);
      if (best_j != j) break;
    }
    n_pre = cs.best_pre.ctas;
  } else {
    cs.best_pre = LevelPlan{};
    cs.best_suf = LevelPlan{};
  }
  *batch_out = batch;
  *n_pre_out = n_pre;
  *span_out = best_span;
  *alpha_out = alpha;
  *floor_s_out = floor_s;
  return PKD_OK;
}

int plan_schedule_cascade(const pkd_config& cfg, int32_t n_cta, const Layout& L,
                          const int32_t* group_indptr, int32_t n_groups,
                          const int32_t* p_indptr, const int32_t* p_indices,
                          const int32_t* p_last, const int32_t* s_indptr,
                          const int32_t* s_indices, const int32_t* s_last, int32_t* words,
                          pkd_plan_info* info) {
  if (words == nullptr) return PKD_E_INVALID_ARG;
  const int64_t P = cfg.page_size;
  const int32_t R = block_rows(cfg);
  const int32_t hkv = cfg.num_kv_heads;
  thread_local Scratch sc;
  thread_local CascadeScratch cs;
  int32_t batch = 0, n_pre = 0;
  int64_t best_span = 0, alpha = 0, floor_s = 0;
  int st = cascade_search(cfg, n_cta, group_indptr, n_groups, p_indptr, p_last, s_indptr, s_last,
                          sc, cs, &batch, &n_pre, &best_span, &alpha, &floor_s);
  if (st != PKD_OK) return st;
  const int64_t nnz_p = n_groups > 0 ? p_indptr[n_groups] : 0;
  const int64_t nnz_s = batch > 0 ? s_indptr[batch] : 0;
  if (nnz_p + nnz_s > cfg.max_num_pages) return PKD_E_CAPACITY;
  if ((nnz_p > 0 && p_indices == nullptr) || (nnz_s > 0 && s_indices == nullptr))
    return PKD_E_INVALID_ARG;
  // page list: the prefix table's indices, then the suffix table's
  if (!copy_checked(p_indices, words + L.page_list, nnz_p, cfg.num_pages) ||
      !copy_checked(s_indices, words + L.page_list + nnz_p, nnz_s, cfg.num_pages))
    return PKD_E_BAD_TABLE;
  int64_t suf_total = 0;
  for (int64_t l : cs.suf_len) suf_total += l;
  const LevelPlan& pre = cs.best_pre;
  const LevelPlan& suf = cs.best_suf;
  const int64_t n_items = (int64_t)pre.items.size() + (int64_t)suf.items.size();
  if (n_items > L.max_items || batch > L.max_items) return PKD_E_CAPACITY;

  // ---- reduction map: every request a unit, prefix chunks then suffix chunks
  const int32_t n_blocks = (int32_t)cs.blocks.size();
  cs.np_block.assign((size_t)n_blocks, 0);
  int64_t max_pchunk = 0;
  for (int32_t b = 0; b < n_blocks; ++b) {
    cs.np_block[b] = (int32_t)ceil_div(cs.block_len[b], pre.block_chunk[b]);
    max_pchunk = std::max(max_pchunk, std::min(pre.block_chunk[b], cs.block_len[b]));
  }
  cs.ns_req.assign((size_t)batch, 0);
  int32_t* merge_indptr = words + L.merge_indptr;
  int32_t* unit_words = words + L.units;
  merge_indptr[0] = 0;
  int32_t max_chunks = 0;
  for (int32_t r = 0; r < batch; ++r) {
    cs.ns_req[r] = (int32_t)ceil_div(cs.suf_len[r], suf.chunk);
    const int32_t n = cs.np_block[cs.block_of[r]] + cs.ns_req[r];
    unit_words[2 * r] = r;
    unit_words[2 * r + 1] = n;
    merge_indptr[r + 1] = merge_indptr[r] + n;
    max_chunks = std::max(max_chunks, n);
  }
  const int64_t n_slots = batch > 0 ? merge_indptr[batch] : 0;
  if (n_slots > L.max_slots) return PKD_E_CAPACITY;

  // ---- queues: prefix items on CTAs [0, n_pre), suffix items after
  cs.count.assign((size_t)n_cta, 0);
  for (int32_t o : pre.owner) cs.count[o]++;
  for (int32_t o : suf.owner) cs.count[n_pre + o]++;
  int32_t* cta_indptr = words + L.cta_indptr;
  cta_indptr[0] = 0;
  for (int32_t c = 0; c < n_cta; ++c) cta_indptr[c + 1] = cta_indptr[c] + cs.count[c];
  cs.fill.assign(cta_indptr, cta_indptr + n_cta);
  int32_t* item_words = words + L.items;
  for (size_t j = 0; j < pre.items.size(); ++j) {
    const Item& it = pre.items[j];
    const Block& bk = cs.blocks[it.req / hkv];
    int32_t* w = item_words + (int64_t)cs.fill[pre.owner[j]]++ * kItemWords;
    w[0] = bk.req_first;
    w[1] = it.tok_begin;
    w[2] = it.tok_end;
    w[3] = it.chunk_idx;                       // slot of request r: merge_indptr[r] + chunk
    w[4] = (int32_t)(p_indptr[bk.table_row] + it.tok_begin / P);
    w[5] = bk.n_req;
    w[6] = -1;                                 // cascade prefix item
    w[7] = it.req % hkv;
  }
  for (size_t j = 0; j < suf.items.size(); ++j) {
    const Item& it = suf.items[j];
    const int32_t r = it.req;
    int32_t* w = item_words + (int64_t)cs.fill[n_pre + suf.owner[j]]++ * kItemWords;
    w[0] = r;
    w[1] = it.tok_begin;
    w[2] = it.tok_end;
    w[3] = merge_indptr[r] + cs.np_block[cs.block_of[r]] + it.chunk_idx;
    w[4] = (int32_t)(nnz_p + s_indptr[r] + it.tok_begin / P);
    w[5] = 1;
    w[6] = 0;
    w[7] = 0;
  }

  int32_t* h = words;
  std::memset(h, 0, sizeof(int32_t) * H_WORDS);
  h[H_MAGIC] = kMagic;
  h[H_BATCH] = batch;
  h[H_HQ] = cfg.num_qo_heads;
  h[H_HKV] = cfg.num_kv_heads;
  h[H_D] = cfg.head_dim;
  h[H_P] = cfg.page_size;
  h[H_NCTA] = n_cta;
  h[H_NITEMS] = (int32_t)n_items;
  h[H_NUNITS] = batch;
  h[H_NSLOTS] = (int32_t)n_slots;
  h[H_CHUNK] = (int32_t)std::max<int64_t>(suf.chunk, 0);
  h[H_ALPHA] = (int32_t)alpha;
  h[H_NNZ] = (int32_t)(nnz_p + nnz_s);
  h[H_MAKESPAN] = (int32_t)std::min<int64_t>(best_span / 16, 0x7fffffff);
  h[H_MINCHUNK] = (int32_t)floor_s;
  h[H_BLOCK] = R;
  h[H_MAXCHUNKS] = max_chunks;
  h[H_MAXBATCH] = cfg.max_batch;
  h[H_MAXPAGES] = cfg.max_num_pages;
  h[H_NPRE] = n_pre;
  h[H_PCHUNK] = (int32_t)max_pchunk;

  if (info) {
    info->batch = batch;
    info->num_ctas = n_cta;
    info->chunk_tokens = h[H_CHUNK];
    info->num_items = (int32_t)n_items;
    info->num_units = batch;
    info->num_slots = (int32_t)n_slots;
    info->total_tokens = suf_total;
    for (const Block& bk : cs.blocks) info->total_tokens += cs.pre_row[bk.table_row] * bk.n_req;
    info->makespan = best_span / 16;
    info->nnz = (int32_t)(nnz_p + nnz_s);
    info->schedule_words = (int32_t)(L.page_list + nnz_p + nnz_s);
    info->prefix_ctas = n_pre;
    info->prefix_chunk_tokens = h[H_PCHUNK];
  }
  return PKD_OK;
}

// ---------------------------------------------------------------- advice
//
// Which format serves a shared-prefix step faster ("FlashInfer 完全拆解",
// Composable Format 只在复用足够大时占优: the split into a shared level only
// pays once the reuse is large enough): the cascade plan (shared prefix once,
// suffixes apart, one merge) or the single format (every request over its
// whole table, prefix pages then its own).  Each is predicted from its own
// planner's makespan M: the cascade search above, and the plain planner's
// chunk choice (candidates L, L/2, L/4 of the work bound, floor 256, alpha
// 32) over the concatenated lengths, and from the KV bytes it reads (the
// prefix once, or once per request).  GPU time per layer = a + b M + c MB
// (steps launched back to back), a least-squares fit on GB300 over the
// pages' grid of shared prefix x batch (1,024 / 8,192 / 32,768 tokens x 16 /
// 64 requests) and prefixes of 16 to 256 tokens, all with 128-token
// suffixes: cascade 5.58 us + 0.02523 us per makespan unit + 0.1143 us per
// MB, single 4.30 us + 0.04393 us per token + 0.00648 us per MB (the
// single format's prefix pages come from L2 for all but the first request).
constexpr double kAdviceCascadeUs0 = 5.58, kAdviceCascadeUsPerUnit = 0.02523,
                 kAdviceCascadeUsPerMB = 0.1143;
constexpr double kAdviceSingleUs0 = 4.30, kAdviceSingleUsPerToken = 0.04393,
                 kAdviceSingleUsPerMB = 0.00648;

// The plain planner's makespan for these lengths (its chunk candidates and
// LPT, without the schedule).
int64_t plain_makespan(const std::vector<int64_t>& lens, int32_t n_cta, int64_t P, Scratch& sc) {
  int64_t total = 0;
  for (int64_t l : lens) total += l;
  if (lens.empty()) return 0;
  const int64_t alpha = kDefaultAlpha;
  const int64_t floor_c = ceil_div(kDefaultMinChunk, P) * P;
  const int64_t bound = ceil_div(total, n_cta);
  int64_t best = -1;
  std::vector<int64_t> seen;
  for (int64_t k : {1, 2, 4}) {
    const int64_t c = std::max(ceil_div(ceil_div(bound, k), P) * P, floor_c);
    if (std::find(seen.begin(), seen.end(), c) != seen.end()) continue;
    seen.push_back(c);
    split_sorted(lens, c, alpha, &sc.whole, &sc.rest, &sc.items);
    const int64_t span = lpt(sc.items, n_cta, &sc.owner, &sc.heap);
    if (best < 0 || span < best) best = span;
  }
  return best;
}

int advise_format(const pkd_config& cfg, int32_t n_cta, const int32_t* group_indptr,
                  int32_t n_groups, const int32_t* p_indptr, const int32_t* p_last,
                  const int32_t* s_indptr, const int32_t* s_last, pkd_format_advice* out) {
  if (out == nullptr) return PKD_E_INVALID_ARG;
  thread_local Scratch sc;
  thread_local CascadeScratch cs;
  int32_t batch = 0, n_pre = 0;
  int64_t span = 0, alpha = 0, floor_s = 0;
  const int st = cascade_search(cfg, n_cta, group_indptr, n_groups, p_indptr, p_last, s_indptr,
                                s_last, sc, cs, &batch, &n_pre, &span, &alpha, &floor_s);
  if (st != PKD_OK) return st;
  std::vector<int64_t> whole((size_t)batch);
  int64_t single_tokens = 0, cascade_tokens = 0;
  for (int32_t r = 0; r < batch; ++r) {
    whole[r] = cs.block_len[cs.block_of[r]] + cs.suf_len[r];
    single_tokens += whole[r];
    cascade_tokens += cs.suf_len[r];
  }
  for (int32_t j = 0; j < n_groups; ++j) cascade_tokens += cs.pre_row[j];
  const double mb_per_token = 2.0 * cfg.num_kv_heads * cfg.head_dim * 2 / 1e6;
  const int64_t ms = plain_makespan(whole, n_cta, cfg.page_size, sc);
  std::memset(out, 0, sizeof(*out));
  out->prefix_ctas = n_pre;
  out->cascade_makespan = span / 16;
  out->single_makespan = ms;
  out->cascade_us = (float)(kAdviceCascadeUs0 + kAdviceCascadeUsPerUnit * (double)(span / 16) +
                            kAdviceCascadeUsPerMB * mb_per_token * (double)cascade_tokens);
  out->single_us = (float)(kAdviceSingleUs0 + kAdviceSingleUsPerToken * (double)ms +
                           kAdviceSingleUsPerMB * mb_per_token * (double)single_tokens);
  out->use_cascade = batch > 0 && out->cascade_us < out->single_us ? 1 : 0;
  return PKD_OK;
}

}  // namespace pkd
