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
  std::vector<int32_t> owner, best_owner, first_slot, n_chunks, count, fill, by_pos;
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
  // one slot per chunk, units in ascending request order, slots in chunk order
  std::vector<int32_t>& first_slot = sc.first_slot;  // slot of the block's first request
  std::vector<int32_t>& n_chunks = sc.n_chunks;
  std::vector<std::pair<int32_t, int32_t>>& units = sc.units;
  first_slot.assign((size_t)n_blocks, -1);
  n_chunks.assign((size_t)n_blocks, 1);
  units.clear();
  int64_t n_slots = 0;
  for (int32_t b = 0; b < n_blocks; ++b) {
    const int64_t nc = ceil_div(lens[b], best_chunk);
    n_chunks[b] = (int32_t)nc;
    if (nc > 1) {
      first_slot[b] = (int32_t)n_slots;
      for (int32_t r = 0; r < blocks[b].n_req; ++r) {
        units.emplace_back(blocks[b].req_first + r, (int32_t)nc);
        n_slots += nc;
      }
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

}  // namespace pkd
