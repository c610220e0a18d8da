// C ABI of libpkd: context, workspace, plan publication, run, merge_states,
// CUDA-graph capture.  Host runtime only; the kernels live in
// decode_kernel.cu and merge_kernels.cu, the scheduler in planner.cpp.
//
// Plan publication follows FlashInfer 完全拆解, 固定指针比固定内容更重要: the
// schedule is written into page-locked host staging and copied with
// cudaMemcpyAsync into fixed offsets of the caller's device workspace, so a
// captured run sees new contents at the same addresses.  Staging is
// double-buffered; an event per buffer keeps a pending copy from being
// overwritten.
#include <cuda_runtime.h>

#include <cmath>
#include <cstring>
#include <new>
#include <vector>

#include "append_layers.h"
#include "pkd_internal.h"

using namespace pkd;

struct KvMapEntry {
  const void* kv = nullptr;
  CUtensorMap map{};
  CUtensorMap map_dense{};   // cascade contexts: the dense role's per-head map too
};

struct pkd_ctx {
  pkd_config cfg;
  int32_t n_cta = 0;
  DecodeKind kind{};   // which decode kernel (consumer, cache type, producer)
  int smem_bytes = 0;
  // page-tile maps by cache address (the map holds only the address and the
  // context's fixed shape), replaced round-robin
  std::vector<KvMapEntry> kv_maps;
  size_t next_map = 0;
  int merge_grid = 0;
  int device = 0;
  Layout layout{};
  uint8_t* ws = nullptr;
  size_t ws_bytes = 0;
  int32_t* staging[2] = {nullptr, nullptr};
  int32_t* err_host = nullptr;   // page-locked landing word of the device error word
  cudaEvent_t staged[2] = {nullptr, nullptr};
  bool staged_pending[2] = {false, false};
  int next_staging = 0;
  uint64_t epoch = 0;
  pkd_plan_info info{};
  int32_t max_chunks = 0;   // header word H_MAXCHUNKS of the published plan
};

struct pkd_graph {
  pkd_ctx* ctx = nullptr;
  int32_t layers = 0;
  int32_t batch = 0;   // the plan's batch at capture (dense-prefix graphs hold q maps of it)
  cudaGraphExec_t exec = nullptr;
  std::vector<cudaEvent_t> ev;  // [2 * layers] when timing
};

namespace {

bool valid_group(int g) { return g == 1 || g == 2 || g == 4 || g == 8; }

// The consumer flags exclude each other; the shared-prefix kernel exists for
// the tensor-core consumer only.
bool valid_flags(uint32_t f) {
  const uint32_t known = PKD_FLAG_FMA_CONSUMER | PKD_FLAG_MMA_CONSUMER | PKD_FLAG_SHARED_PREFIX |
                         PKD_FLAG_KV_FP8 | PKD_FLAG_ROW_COPIES | PKD_FLAG_CHUNK_SEARCH |
                         PKD_FLAG_HND | PKD_FLAG_DENSE_PREFIX | PKD_FLAG_CASCADE;
  if (f & ~known) return false;
  // a cascade context runs both of its levels itself: bf16 page tiles,
  // tensor cores, either layout
  if ((f & PKD_FLAG_CASCADE) && (f & ~(PKD_FLAG_CASCADE | PKD_FLAG_MMA_CONSUMER | PKD_FLAG_HND)))
    return false;
  if ((f & PKD_FLAG_FMA_CONSUMER) &&
      (f & (PKD_FLAG_MMA_CONSUMER | PKD_FLAG_SHARED_PREFIX | PKD_FLAG_KV_FP8)))
    return false;
  if ((f & PKD_FLAG_SHARED_PREFIX) && (f & PKD_FLAG_KV_FP8)) return false;
  // the dense-prefix kernel: shared-prefix plans, tensor cores, bf16 page tiles
  if ((f & PKD_FLAG_DENSE_PREFIX) &&
      (!(f & PKD_FLAG_SHARED_PREFIX) ||
       (f & (PKD_FLAG_FMA_CONSUMER | PKD_FLAG_KV_FP8 | PKD_FLAG_ROW_COPIES))))
    return false;
  return true;
}

int check_config(const pkd_config* c) {
  if (c == nullptr) return PKD_E_INVALID_ARG;
  if (!valid_flags(c->flags)) return PKD_E_INVALID_ARG;
  if (c->max_batch < 0 || c->max_num_pages < 0 || c->num_pages < 1 || c->page_size < 1 ||
      c->num_ctas < 0)
    return PKD_E_INVALID_ARG;
  if (c->head_dim != kHeadDim) return PKD_E_UNSUPPORTED_SHAPE;
  if (c->num_kv_heads < 1 || c->num_kv_heads > kMaxKvHeads) return PKD_E_UNSUPPORTED_SHAPE;
  if (c->num_qo_heads < 1 || c->num_qo_heads % c->num_kv_heads != 0)
    return PKD_E_UNSUPPORTED_SHAPE;
  if (!valid_group(c->num_qo_heads / c->num_kv_heads)) return PKD_E_UNSUPPORTED_SHAPE;
  // the dense-prefix kernel (and the cascade kernel) read 16-token page tiles
  if ((c->flags & (PKD_FLAG_DENSE_PREFIX | PKD_FLAG_CASCADE)) && c->page_size % 16 != 0)
    return PKD_E_UNSUPPORTED_SHAPE;
  // a page must fit the copy-size and tx-count limits of one stage
  if ((int64_t)c->page_size * c->num_kv_heads * kHeadDim * 2 * 2 > (int64_t)1 << 30)
    return PKD_E_UNSUPPORTED_SHAPE;
  return PKD_OK;
}

// The decode kernel a configuration selects.  Page tiles need a page size
// that is a multiple of the 16-token box, a tensor-core consumer, and a
// driver that encodes the map (checked on `probe_address`, a device address
// standing in for the cache -- encoding records the address and checks the
// shape; with a null probe the check is skipped).
DecodeKind kind_for(const pkd_config* c, const void* probe_address) {
  DecodeKind k;
  k.group = c->num_qo_heads / c->num_kv_heads;
  k.mma = use_mma_consumer(k.group, c->flags);
  k.block = (c->flags & PKD_FLAG_SHARED_PREFIX) != 0;
  k.fp8 = (c->flags & PKD_FLAG_KV_FP8) != 0;
  k.tmap = k.mma && c->page_size % 16 == 0 && !(c->flags & PKD_FLAG_ROW_COPIES);
  k.dense = (c->flags & PKD_FLAG_DENSE_PREFIX) != 0;
  k.cascade = (c->flags & PKD_FLAG_CASCADE) != 0;
  if (k.tmap && probe_address != nullptr) {
    CUtensorMap m;
    const bool hnd = (c->flags & PKD_FLAG_HND) != 0;
    k.tmap = encode_kv_map(probe_address, c->num_pages, c->page_size, c->num_kv_heads, k.fp8,
                           hnd, k.dense, &m) == cudaSuccess;
    if (k.cascade)   // the cascade kernel needs the dense role's map too
      k.tmap = k.tmap && encode_kv_map(probe_address, c->num_pages, c->page_size,
                                       c->num_kv_heads, false, hnd, true, &m) == cudaSuccess;
  }
  return k;
}

int resolve_ctas(const pkd_config* c, const DecodeKind& k, int32_t* n_cta, int* smem_bytes) {
  *smem_bytes = decode_smem_bytes(c->num_kv_heads, k);
  if (c->num_ctas > 0) {
    *n_cta = c->num_ctas;
    return PKD_OK;
  }
  int dev = 0, sms = 0, per_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKD_E_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return PKD_E_CUDA;
  if (decode_prepare(k, *smem_bytes) != cudaSuccess) return PKD_E_CUDA;
  if (decode_occupancy(k, c->num_kv_heads, *smem_bytes, &per_sm) != cudaSuccess)
    return PKD_E_CUDA;
  if (per_sm < 1) return PKD_E_UNSUPPORTED_SHAPE;
  *n_cta = sms * per_sm;
  return PKD_OK;
}

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

// The page-tile map(s) of the cache at kv (cached per address).
int kv_map_for(pkd_ctx* ctx, const void* kv, CUtensorMap* out, CUtensorMap* out_dense = nullptr) {
  for (const KvMapEntry& e : ctx->kv_maps)
    if (e.kv == kv) {
      *out = e.map;
      if (out_dense) *out_dense = e.map_dense;
      return PKD_OK;
    }
  KvMapEntry e;
  e.kv = kv;
  const pkd_config& c = ctx->cfg;
  const bool hnd = (c.flags & PKD_FLAG_HND) != 0;
  if (encode_kv_map(kv, c.num_pages, c.page_size, c.num_kv_heads, ctx->kind.fp8, hnd,
                    ctx->kind.dense, &e.map) != cudaSuccess)
    return PKD_E_CUDA;
  if (ctx->kind.cascade &&
      encode_kv_map(kv, c.num_pages, c.page_size, c.num_kv_heads, false, hnd, true,
                    &e.map_dense) != cudaSuccess)
    return PKD_E_CUDA;
  constexpr size_t kMaxMaps = 128;
  if (ctx->kv_maps.size() < kMaxMaps) {
    ctx->kv_maps.push_back(e);
  } else {
    ctx->kv_maps[ctx->next_map] = e;
    ctx->next_map = (ctx->next_map + 1) % kMaxMaps;
  }
  *out = e.map;
  if (out_dense) *out_dense = e.map_dense;
  return PKD_OK;
}

int launch_run(pkd_ctx* ctx, const void* q, const void* kv, void* out, float* lse,
               float k_scale, float v_scale, cudaStream_t stream, cudaEvent_t ev_before,
               cudaEvent_t ev_after, int32_t wait_epoch = 0) {
  const pkd_config& c = ctx->cfg;
  DecodeArgs a{};
  a.wait_epoch = wait_epoch;
  a.sched = reinterpret_cast<const int32_t*>(ctx->ws);
  a.o_part = reinterpret_cast<float*>(ctx->ws + ctx->layout.o_part_byte);
  a.l_part = reinterpret_cast<float*>(ctx->ws + ctx->layout.l_part_byte);
  a.err = reinterpret_cast<int32_t*>(ctx->ws + ctx->layout.err_byte);
  a.q = static_cast<const uint16_t*>(q);
  a.kv = static_cast<const uint8_t*>(kv);
  a.out = static_cast<uint16_t*>(out);
  a.lse = lse;
  a.row_bytes = c.num_kv_heads * kHeadDim * (ctx->kind.fp8 ? 1 : 2);
  a.page_bytes = (int64_t)2 * c.page_size * a.row_bytes;
  a.off_cta = ctx->layout.cta_indptr;
  a.off_items = ctx->layout.items;
  a.off_pages = ctx->layout.page_list;
  a.off_merge = ctx->layout.merge_indptr;
  a.hq = c.num_qo_heads;
  a.hkv = c.num_kv_heads;
  a.page_size = c.page_size;
  a.num_pages = c.num_pages;
  a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)c.head_dim) * (double)k_scale);
  a.v_scale = v_scale;
  // page size 1: HND and NHD are the same bytes, and a token's K and V rows
  // are adjacent (one copy moves both)
  a.hnd = ((c.flags & PKD_FLAG_HND) && c.page_size > 1) ? 1 : 0;
  a.kv_merged = (c.page_size == 1 && !ctx->kind.tmap) ? 1 : 0;
  CascadeArgs ca{};
  if (ctx->kind.tmap && kv != nullptr) {
    const int st = kv_map_for(ctx, kv, &a.kv_map, ctx->kind.cascade ? &ca.pre.kv_map : nullptr);
    if (st != PKD_OK) return st;
  }
  if ((ctx->kind.dense || ctx->kind.cascade) && ctx->info.batch > 0 &&
      encode_q_map(q, ctx->info.batch, c.num_qo_heads, c.num_kv_heads, &a.q_map) != cudaSuccess)
    return PKD_E_CUDA;
  if (ev_before && cudaEventRecordWithFlags(ev_before, stream, cudaEventRecordExternal) != cudaSuccess)
    return PKD_E_CUDA;
  if (ctx->kind.cascade) {
    // the suffix role: a's all-heads map; the prefix role: the same
    // arguments with the dense per-head map (and a's query map)
    const CUtensorMap dense_map = ca.pre.kv_map;
    ca.suf = a;
    ca.pre = a;
    ca.pre.kv_map = dense_map;
    if (launch_cascade(ctx->kind, ca, ctx->n_cta, c.num_kv_heads, ctx->smem_bytes, stream) !=
        cudaSuccess)
      return PKD_E_CUDA;
  } else if (launch_decode(ctx->kind, a, ctx->n_cta, c.num_kv_heads, ctx->smem_bytes, stream) !=
             cudaSuccess) {
    return PKD_E_CUDA;
  }
  if (ev_after && cudaEventRecordWithFlags(ev_after, stream, cudaEventRecordExternal) != cudaSuccess)
    return PKD_E_CUDA;
  MergeArgs m{};
  m.sched = a.sched;
  m.o_part = a.o_part;
  m.l_part = a.l_part;
  m.out = a.out;
  m.lse = lse;
  m.off_units = ctx->layout.units;
  m.off_merge = ctx->layout.merge_indptr;
  m.hq = c.num_qo_heads;
  m.wait_epoch = wait_epoch;
  if (launch_merge_partials(m, ctx->merge_grid, ctx->max_chunks, stream,
                            ctx->kind.cascade) != cudaSuccess)
    return PKD_E_CUDA;
  return PKD_OK;
}

}  // namespace

extern "C" {

int pkd_version(void) { return 100; }

const char* pkd_status_str(int s) {
  switch (s) {
    case PKD_OK: return "ok";
    case PKD_E_INVALID_ARG: return "invalid argument";
    case PKD_E_BAD_TABLE: return "bad page table (indptr / indices / last_page_len)";
    case PKD_E_UNSUPPORTED_SHAPE: return "unsupported shape";
    case PKD_E_WORKSPACE_TOO_SMALL: return "workspace too small";
    case PKD_E_NO_PLAN: return "run before plan";
    case PKD_E_STALE_PLAN: return "stale plan (epoch mismatch)";
    case PKD_E_CAPACITY: return "batch or page count above the configured capacity";
    case PKD_E_CUDA: return "CUDA runtime error";
    case PKD_E_DEVICE: return "device error word set";
    case PKD_E_SCRATCH_LIMIT: return "layout larger than the static scratch array (32 MiB)";
    default: return "unknown status";
  }
}

int pkd_schedule_layout(const pkd_config* cfg, int64_t off[6]) {
  if (off == nullptr) return PKD_E_INVALID_ARG;
  int st = check_config(cfg);
  if (st != PKD_OK) return st;
  if (cfg->num_ctas < 1) return PKD_E_INVALID_ARG;
  Layout L = make_layout(*cfg, cfg->num_ctas);
  off[0] = L.cta_indptr;
  off[1] = L.items;
  off[2] = L.units;
  off[3] = L.merge_indptr;
  off[4] = L.page_list;
  off[5] = L.words;
  return PKD_OK;
}

int pkd_plan_host_shared(const pkd_config* cfg, const int32_t* group_indptr, int32_t num_groups,
                         const int32_t* indptr, const int32_t* indices,
                         const int32_t* last_page_len, int32_t* host_words, size_t max_words,
                         pkd_plan_info* info) {
  int st = check_config(cfg);
  if (st != PKD_OK) return st;
  if (cfg->num_ctas < 1 || host_words == nullptr || !(cfg->flags & PKD_FLAG_SHARED_PREFIX))
    return PKD_E_INVALID_ARG;
  if (num_groups > 0 && group_indptr == nullptr) return PKD_E_INVALID_ARG;
  Layout L = make_layout(*cfg, cfg->num_ctas);
  if (max_words < (size_t)L.words) return PKD_E_INVALID_ARG;
  return plan_schedule_grouped(*cfg, cfg->num_ctas, L, group_indptr, num_groups, indptr, indices,
                               last_page_len, host_words, info);
}

int pkd_plan_host_cascade(const pkd_config* cfg, const int32_t* group_indptr,
                          int32_t num_groups, const int32_t* p_indptr, const int32_t* p_indices,
                          const int32_t* p_last, const int32_t* s_indptr,
                          const int32_t* s_indices, const int32_t* s_last, int32_t* host_words,
                          size_t max_words, pkd_plan_info* info) {
  int st = check_config(cfg);
  if (st != PKD_OK) return st;
  if (cfg->num_ctas < 2 || host_words == nullptr || !(cfg->flags & PKD_FLAG_CASCADE))
    return PKD_E_INVALID_ARG;
  Layout L = make_layout(*cfg, cfg->num_ctas);
  if (max_words < (size_t)L.words) return PKD_E_INVALID_ARG;
  return plan_schedule_cascade(*cfg, cfg->num_ctas, L, group_indptr, num_groups, p_indptr,
                               p_indices, p_last, s_indptr, s_indices, s_last, host_words, info);
}

int pkd_advise_format(const pkd_config* cfg, const int32_t* group_indptr, int32_t num_groups,
                      const int32_t* p_indptr, const int32_t* p_last, const int32_t* s_indptr,
                      const int32_t* s_last, pkd_format_advice* advice) {
  int st = check_config(cfg);
  if (st != PKD_OK) return st;
  if (cfg->num_ctas < 2 || advice == nullptr || !(cfg->flags & PKD_FLAG_CASCADE))
    return PKD_E_INVALID_ARG;
  return advise_format(*cfg, cfg->num_ctas, group_indptr, num_groups, p_indptr, p_last, s_indptr,
                       s_last, advice);
}

int pkd_plan_host(const pkd_config* cfg, const int32_t* indptr, const int32_t* indices,
                  const int32_t* last_page_len, int32_t batch, int32_t* host_words,
                  size_t max_words, pkd_plan_info* info) {
  int st = check_config(cfg);
  if (st != PKD_OK) return st;
  if (cfg->num_ctas < 1 || host_words == nullptr || (cfg->flags & PKD_FLAG_CASCADE))
    return PKD_E_INVALID_ARG;
  Layout L = make_layout(*cfg, cfg->num_ctas);
  if (max_words < (size_t)L.words) return PKD_E_INVALID_ARG;
  return plan_schedule(*cfg, cfg->num_ctas, L, indptr, indices, last_page_len, batch,
                       host_words, info);
}

size_t pkd_workspace_bytes(const pkd_config* cfg) {
  if (check_config(cfg) != PKD_OK) return 0;
  int32_t n_cta = 0;
  int smem = 0;
  // the workspace layout does not depend on the producer
  if (resolve_ctas(cfg, kind_for(cfg, nullptr), &n_cta, &smem) != PKD_OK) return 0;
  return make_layout(*cfg, n_cta).total_bytes;
}

int pkd_create(const pkd_config* cfg, void* d_workspace, size_t workspace_bytes,
               pkd_ctx** out) {
  if (out == nullptr) return PKD_E_INVALID_ARG;
  *out = nullptr;
  int st = check_config(cfg);
  if (st != PKD_OK) return st;
  if (d_workspace == nullptr || !aligned(d_workspace, 256)) return PKD_E_INVALID_ARG;
  pkd_ctx* ctx = new (std::nothrow) pkd_ctx();
  if (!ctx) return PKD_E_INVALID_ARG;
  ctx->cfg = *cfg;
  ctx->kind = kind_for(cfg, d_workspace);
  if ((ctx->kind.dense || ctx->kind.cascade) && !ctx->kind.tmap) {   // the driver refused a map
    delete ctx;
    return PKD_E_UNSUPPORTED_SHAPE;
  }
  st = resolve_ctas(cfg, ctx->kind, &ctx->n_cta, &ctx->smem_bytes);
  if (st != PKD_OK) {
    delete ctx;
    return st;
  }
  if (decode_prepare(ctx->kind, ctx->smem_bytes) != cudaSuccess) {
    delete ctx;
    return PKD_E_CUDA;
  }
  ctx->layout = make_layout(*cfg, ctx->n_cta);
  if (workspace_bytes < ctx->layout.total_bytes) {
    delete ctx;
    return PKD_E_WORKSPACE_TOO_SMALL;
  }
  cudaGetDevice(&ctx->device);
  ctx->merge_grid = merge_grid_for(ctx->n_cta);
  ctx->ws = static_cast<uint8_t*>(d_workspace);
  ctx->ws_bytes = workspace_bytes;
  for (int k = 0; k < 2; ++k) {
    if (cudaMallocHost(&ctx->staging[k], (size_t)ctx->layout.words * 4) != cudaSuccess ||
        cudaEventCreateWithFlags(&ctx->staged[k], cudaEventDisableTiming) != cudaSuccess) {
      pkd_destroy(ctx);
      return PKD_E_CUDA;
    }
    std::memset(ctx->staging[k], 0, (size_t)ctx->layout.words * 4);
  }
  if (cudaMallocHost(&ctx->err_host, sizeof(int32_t)) != cudaSuccess) {
    pkd_destroy(ctx);
    return PKD_E_CUDA;
  }
  *ctx->err_host = 0;
  if (cudaMemset(ctx->ws + ctx->layout.err_byte, 0, 4) != cudaSuccess ||
      cudaDeviceSynchronize() != cudaSuccess) {
    pkd_destroy(ctx);
    return PKD_E_CUDA;
  }
  *out = ctx;
  return PKD_OK;
}

void pkd_destroy(pkd_ctx* ctx) {
  if (!ctx) return;
  for (int k = 0; k < 2; ++k) {
    if (ctx->staged[k]) {
      cudaEventSynchronize(ctx->staged[k]);
      cudaEventDestroy(ctx->staged[k]);
    }
    if (ctx->staging[k]) cudaFreeHost(ctx->staging[k]);
  }
  if (ctx->err_host) cudaFreeHost(ctx->err_host);
  delete ctx;
}

}  // extern "C"

// Plan into the next staging buffer (plan_fn(words, info) runs the planner)
// and publish it.
template <typename PlanFn>
static int plan_and_publish(pkd_ctx* ctx, PlanFn plan_fn, void* stream, uint64_t* epoch) {
  if (ctx == nullptr) return PKD_E_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int k = ctx->next_staging;
  if (ctx->staged_pending[k]) {
    if (cudaEventSynchronize(ctx->staged[k]) != cudaSuccess) return PKD_E_CUDA;
    ctx->staged_pending[k] = false;
  }
  int32_t* words = ctx->staging[k];
  pkd_plan_info info{};
  int st = plan_fn(words, &info);
  if (st != PKD_OK) return st;
  const Layout& L = ctx->layout;
  // two copies in stream order: first the body (cta queues, items, units,
  // merge map and the page list behind them, as laid out in the workspace),
  // then the header with the plan's epoch word, so that a kernel that sees
  // the new epoch (a run on another stream, pkd_run with expect_epoch) also
  // sees the whole schedule
  words[H_EPOCH] = epoch_word(ctx->epoch + 1);
  if (cudaMemcpyAsync(ctx->ws + (size_t)H_WORDS * 4, words + H_WORDS,
                      ((size_t)L.page_list + (size_t)info.nnz - H_WORDS) * 4,
                      cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(ctx->ws, words, (size_t)H_WORDS * 4, cudaMemcpyHostToDevice, s) !=
          cudaSuccess)
    return PKD_E_CUDA;
  if (cudaEventRecord(ctx->staged[k], s) != cudaSuccess) return PKD_E_CUDA;
  ctx->staged_pending[k] = true;
  ctx->next_staging = k ^ 1;
  info.page_tiles = ctx->kind.tmap ? 1 : 0;
  ctx->info = info;
  ctx->max_chunks = words[H_MAXCHUNKS];
  ctx->epoch += 1;
  if (epoch) *epoch = ctx->epoch;
  return PKD_OK;
}

extern "C" {

int pkd_plan(pkd_ctx* ctx, const int32_t* indptr, const int32_t* indices,
             const int32_t* last_page_len, int32_t batch, void* stream, uint64_t* epoch) {
  if (ctx == nullptr || ctx->kind.cascade) return PKD_E_INVALID_ARG;
  return plan_and_publish(
      ctx,
      [&](int32_t* words, pkd_plan_info* info) {
        return plan_schedule_grouped(ctx->cfg, ctx->n_cta, ctx->layout, nullptr, batch, indptr,
                                     indices, last_page_len, words, info);
      },
      stream, epoch);
}

int pkd_plan_shared(pkd_ctx* ctx, const int32_t* group_indptr, int32_t num_groups,
                    const int32_t* indptr, const int32_t* indices, const int32_t* last_page_len,
                    void* stream, uint64_t* epoch) {
  if (ctx == nullptr || !ctx->kind.block) return PKD_E_INVALID_ARG;
  if (num_groups > 0 && group_indptr == nullptr) return PKD_E_INVALID_ARG;
  return plan_and_publish(
      ctx,
      [&](int32_t* words, pkd_plan_info* info) {
        return plan_schedule_grouped(ctx->cfg, ctx->n_cta, ctx->layout, group_indptr, num_groups,
                                     indptr, indices, last_page_len, words, info);
      },
      stream, epoch);
}

int pkd_plan_cascade(pkd_ctx* ctx, const int32_t* group_indptr, int32_t num_groups,
                     const int32_t* p_indptr, const int32_t* p_indices, const int32_t* p_last,
                     const int32_t* s_indptr, const int32_t* s_indices, const int32_t* s_last,
                     void* stream, uint64_t* epoch) {
  if (ctx == nullptr || !ctx->kind.cascade) return PKD_E_INVALID_ARG;
  return plan_and_publish(
      ctx,
      [&](int32_t* words, pkd_plan_info* info) {
        return plan_schedule_cascade(ctx->cfg, ctx->n_cta, ctx->layout, group_indptr, num_groups,
                                     p_indptr, p_indices, p_last, s_indptr, s_indices, s_last,
                                     words, info);
      },
      stream, epoch);
}

int pkd_get_plan_info(const pkd_ctx* ctx, pkd_plan_info* info) {
  if (ctx == nullptr || info == nullptr) return PKD_E_INVALID_ARG;
  if (ctx->epoch == 0) return PKD_E_NO_PLAN;
  *info = ctx->info;
  return PKD_OK;
}

int pkd_run(pkd_ctx* ctx, const void* q, const void* kv, void* out, float* lse,
            uint64_t expect_epoch, void* stream) {
  return pkd_run_scaled(ctx, q, kv, out, lse, 1.f, 1.f, expect_epoch, stream);
}

int pkd_run_scaled(pkd_ctx* ctx, const void* q, const void* kv, void* out, float* lse,
                   float k_scale, float v_scale, uint64_t expect_epoch, void* stream) {
  if (!std::isfinite(k_scale) || !std::isfinite(v_scale)) return PKD_E_INVALID_ARG;
  if (ctx == nullptr) return PKD_E_INVALID_ARG;
  if (ctx->epoch == 0) return PKD_E_NO_PLAN;
  if (expect_epoch != 0 && expect_epoch != ctx->epoch) return PKD_E_STALE_PLAN;
  if (ctx->info.batch > 0) {
    if (q == nullptr || kv == nullptr || out == nullptr) return PKD_E_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(kv, 16) || !aligned(out, 16) || !aligned(lse, 4))
      return PKD_E_INVALID_ARG;
  }
  return launch_run(ctx, q, kv, out, lse, k_scale, v_scale, static_cast<cudaStream_t>(stream),
                    nullptr, nullptr, expect_epoch != 0 ? epoch_word(expect_epoch) : 0);
}

int pkd_merge_states(const void* v_a, const float* s_a, const void* v_b, const float* s_b,
                     void* v_out, float* s_out, int32_t n, int32_t heads, int32_t head_dim,
                     void* stream) {
  if (n < 0 || heads < 0 || head_dim < 8 || head_dim % 8 != 0 || head_dim / 8 > 256)
    return PKD_E_INVALID_ARG;
  const int64_t rows = (int64_t)n * heads;
  if (rows == 0) return PKD_OK;
  if (!v_a || !s_a || !v_b || !s_b || !v_out || !s_out) return PKD_E_INVALID_ARG;
  if (!aligned(v_a, 16) || !aligned(v_b, 16) || !aligned(v_out, 16) || !aligned(s_a, 4) ||
      !aligned(s_b, 4) || !aligned(s_out, 4))
    return PKD_E_INVALID_ARG;
  if (launch_merge_states(v_a, s_a, v_b, s_b, v_out, s_out, rows, head_dim,
                          static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return PKD_E_CUDA;
  return PKD_OK;
}

int pkd_append_kv(const void* k_new, const void* v_new, const int32_t* batch_indices,
                  const int32_t* positions, int32_t n, const int32_t* indptr,
                  const int32_t* indices, const int32_t* last_page_len, int32_t batch, void* kv,
                  int32_t num_pages, int32_t page_size, int32_t num_kv_heads, int32_t head_dim,
                  int32_t* err, void* stream) {
  return pkd_append_kv_ex(k_new, v_new, batch_indices, positions, n, indptr, indices,
                          last_page_len, batch, kv, num_pages, page_size, num_kv_heads, head_dim,
                          0u, err, stream);
}

int pkd_append_kv_ex(const void* k_new, const void* v_new, const int32_t* batch_indices,
                     const int32_t* positions, int32_t n, const int32_t* indptr,
                     const int32_t* indices, const int32_t* last_page_len, int32_t batch,
                     void* kv, int32_t num_pages, int32_t page_size, int32_t num_kv_heads,
                     int32_t head_dim, uint32_t flags, int32_t* err, void* stream) {
  if ((flags & ~(PKD_FLAG_HND | PKD_FLAG_KV_FP8)) != 0) return PKD_E_INVALID_ARG;
  const int elem = (flags & PKD_FLAG_KV_FP8) ? 1 : 2;
  if (n < 0 || batch < 0 || num_pages < 1 || page_size < 1 || num_kv_heads < 1 ||
      head_dim < 1 || ((int64_t)head_dim * elem) % 16 != 0)
    return PKD_E_INVALID_ARG;
  if (n == 0) return PKD_OK;
  if (!k_new || !v_new || !batch_indices || !positions || !indptr || !indices ||
      !last_page_len || !kv)
    return PKD_E_INVALID_ARG;
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(kv, 16) || !aligned(err, 4))
    return PKD_E_INVALID_ARG;
  const int64_t head_bytes = (int64_t)head_dim * elem;
  if (head_bytes * num_kv_heads > (1 << 24)) return PKD_E_INVALID_ARG;
  if (launch_append(k_new, v_new, batch_indices, positions, n, indptr, indices, last_page_len,
                    batch, kv, num_pages, page_size, num_kv_heads, (int32_t)head_bytes,
                    (flags & PKD_FLAG_HND) != 0, err,
                    static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return PKD_E_CUDA;
  return PKD_OK;
}

int pkd_append_kv_layers(int32_t layers, const void* const* k_new, const void* const* v_new,
                         void* const* kv, const int32_t* batch_indices, const int32_t* positions,
                         int32_t n, const int32_t* indptr, const int32_t* indices,
                         const int32_t* last_page_len, int32_t batch, int32_t num_pages,
                         int32_t page_size, int32_t num_kv_heads, int32_t head_dim,
                         uint32_t flags, int32_t* err, void* stream) {
  if ((flags & ~(PKD_FLAG_HND | PKD_FLAG_KV_FP8)) != 0) return PKD_E_INVALID_ARG;
  if (layers < 1 || layers > kMaxAppendLayers || !k_new || !v_new || !kv)
    return PKD_E_INVALID_ARG;
  const int elem = (flags & PKD_FLAG_KV_FP8) ? 1 : 2;
  if (n < 0 || batch < 0 || num_pages < 1 || page_size < 1 || num_kv_heads < 1 ||
      head_dim < 1 || ((int64_t)head_dim * elem) % 16 != 0)
    return PKD_E_INVALID_ARG;
  if (n == 0) return PKD_OK;
  if (!batch_indices || !positions || !indptr || !indices || !last_page_len || !aligned(err, 4))
    return PKD_E_INVALID_ARG;
  const int64_t head_bytes = (int64_t)head_dim * elem;
  if (head_bytes * num_kv_heads > (1 << 24)) return PKD_E_INVALID_ARG;
  AppendLayers L{};
  for (int32_t l = 0; l < layers; ++l) {
    if (!k_new[l] || !v_new[l] || !kv[l] || !aligned(k_new[l], 16) || !aligned(v_new[l], 16) ||
        !aligned(kv[l], 16))
      return PKD_E_INVALID_ARG;
    L.k_new[l] = k_new[l];
    L.v_new[l] = v_new[l];
    L.kv[l] = kv[l];
  }
  if (launch_append_layers(L, layers, batch_indices, positions, n, indptr, indices,
                           last_page_len, batch, num_pages, page_size, num_kv_heads,
                           (int32_t)head_bytes, (flags & PKD_FLAG_HND) != 0, err,
                           static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return PKD_E_CUDA;
  return PKD_OK;
}

int pkd_last_device_error(pkd_ctx* ctx, void* stream, int32_t* dev_err) {
  if (ctx == nullptr || dev_err == nullptr) return PKD_E_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // read, then reset, both behind the stream's work; wait for this stream only
  uint8_t* word = ctx->ws + ctx->layout.err_byte;
  if (cudaMemcpyAsync(ctx->err_host, word, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return PKD_E_CUDA;
  if (cudaMemsetAsync(word, 0, 4, s) != cudaSuccess) return PKD_E_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return PKD_E_CUDA;
  *dev_err = *ctx->err_host;
  return PKD_OK;
}

int pkd_read_schedule(pkd_ctx* ctx, int32_t* host_words, size_t max_words, void* stream) {
  if (ctx == nullptr || host_words == nullptr) return PKD_E_INVALID_ARG;
  if (ctx->epoch == 0) return PKD_E_NO_PLAN;
  const size_t words = (size_t)ctx->layout.page_list + (size_t)ctx->info.nnz;
  if (max_words < words) return PKD_E_INVALID_ARG;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return PKD_E_CUDA;
  if (cudaMemcpy(host_words, ctx->ws, words * 4, cudaMemcpyDeviceToHost) != cudaSuccess)
    return PKD_E_CUDA;
  return PKD_OK;
}

int pkd_graph_capture(pkd_ctx* ctx, int32_t layers, const void* const* q, const void* const* kv,
                      void* const* out, float* const* lse, const float* kv_scales,
                      uint32_t flags, pkd_graph** graph) {
  return pkd_graph_capture_io(ctx, layers, q, kv, out, lse, kv_scales, nullptr, nullptr, nullptr,
                              flags, graph);
}

int pkd_graph_capture_io(pkd_ctx* ctx, int32_t layers, const void* const* q,
                         const void* const* kv, void* const* out, float* const* lse,
                         const float* kv_scales, const void* const* q_host,
                         void* const* out_host, float* const* lse_host, uint32_t flags,
                         pkd_graph** graph) {
  if (ctx == nullptr || graph == nullptr || layers < 1 || q == nullptr || kv == nullptr ||
      out == nullptr)
    return PKD_E_INVALID_ARG;
  if (lse_host != nullptr && lse == nullptr) return PKD_E_INVALID_ARG;
  if ((flags & ~PKD_GRAPH_TIMING) != 0) return PKD_E_INVALID_ARG;
  *graph = nullptr;
  if (ctx->epoch == 0) return PKD_E_NO_PLAN;
  for (int l = 0; l < layers; ++l) {
    if (!q[l] || !kv[l] || !out[l] || !aligned(q[l], 16) || !aligned(kv[l], 16) ||
        !aligned(out[l], 16) || (lse && !aligned(lse[l], 4)))
      return PKD_E_INVALID_ARG;
    if ((q_host && !q_host[l]) || (out_host && !out_host[l]) || (lse_host && !lse_host[l]))
      return PKD_E_INVALID_ARG;
  }
  const pkd_config& c = ctx->cfg;
  const size_t rows = (size_t)ctx->info.batch * c.num_qo_heads;
  const size_t q_bytes = rows * c.head_dim * 2, lse_bytes = rows * 4;
  const bool copy_in = q_host != nullptr && rows > 0;
  const bool copy_out = (out_host != nullptr || lse_host != nullptr) && rows > 0;
  pkd_graph* g = new (std::nothrow) pkd_graph();
  if (!g) return PKD_E_INVALID_ARG;
  g->ctx = ctx;
  g->layers = layers;
  g->batch = ctx->info.batch;
  const bool timing = (flags & PKD_GRAPH_TIMING) != 0;
  if (timing) {
    g->ev.assign((size_t)2 * layers, nullptr);
    for (auto& e : g->ev) {
      if (cudaEventCreate(&e) != cudaSuccess) {
        pkd_graph_destroy(g);
        return PKD_E_CUDA;
      }
    }
  }
  // main capture stream, plus one stream for the query copies and one for
  // the result copies (forked from the main stream, joined before the end);
  // fork / join events exist only while capturing
  cudaStream_t cs = nullptr, cin = nullptr, cout = nullptr;
  std::vector<cudaEvent_t> evs;
  auto new_event = [&evs]() -> cudaEvent_t {
    cudaEvent_t e = nullptr;
    if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return nullptr;
    evs.push_back(e);
    return e;
  };
  int st = PKD_OK;
  if (cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) != cudaSuccess ||
      (copy_in && cudaStreamCreateWithFlags(&cin, cudaStreamNonBlocking) != cudaSuccess) ||
      (copy_out && cudaStreamCreateWithFlags(&cout, cudaStreamNonBlocking) != cudaSuccess))
    st = PKD_E_CUDA;
  cudaEvent_t fork = nullptr;
  std::vector<cudaEvent_t> q_ready, done;
  if (st == PKD_OK) {
    fork = new_event();
    for (int l = 0; l < layers; ++l) {
      q_ready.push_back(copy_in ? new_event() : nullptr);
      done.push_back(copy_out ? new_event() : nullptr);
    }
    if (!fork || (copy_in && !q_ready.back()) || (copy_out && !done.back())) st = PKD_E_CUDA;
  }
  cudaEvent_t in_end = st == PKD_OK && copy_in ? new_event() : nullptr;
  cudaEvent_t out_end = st == PKD_OK && copy_out ? new_event() : nullptr;
  if ((copy_in && !in_end) || (copy_out && !out_end)) st = PKD_E_CUDA;
  cudaGraph_t graph_def = nullptr;
  if (st == PKD_OK && cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal) != cudaSuccess)
    st = PKD_E_CUDA;
  else if (st == PKD_OK) {
    auto ok = [&st](cudaError_t e) {
      if (e != cudaSuccess && st == PKD_OK) st = PKD_E_CUDA;
      return st == PKD_OK;
    };
    ok(cudaEventRecord(fork, cs));
    if (copy_in && ok(cudaStreamWaitEvent(cin, fork, 0))) {
      for (int l = 0; l < layers && st == PKD_OK; ++l) {
        // q[l] is the caller's device query buffer: the copy refills it
        ok(cudaMemcpyAsync(const_cast<void*>(q[l]), q_host[l], q_bytes, cudaMemcpyHostToDevice,
                           cin));
        ok(cudaEventRecord(q_ready[l], cin));
      }
    }
    if (copy_out) ok(cudaStreamWaitEvent(cout, fork, 0));
    for (int l = 0; l < layers && st == PKD_OK; ++l) {
      if (copy_in && !ok(cudaStreamWaitEvent(cs, q_ready[l], 0))) break;
      const float ks = kv_scales ? kv_scales[2 * l] : 1.f;
      const float vs = kv_scales ? kv_scales[2 * l + 1] : 1.f;
      const int r = launch_run(ctx, q[l], kv[l], out[l], lse ? lse[l] : nullptr, ks, vs, cs,
                               timing ? g->ev[2 * l] : nullptr,
                               timing ? g->ev[2 * l + 1] : nullptr);
      if (r != PKD_OK) {
        st = r;
        break;
      }
      if (copy_out && ok(cudaEventRecord(done[l], cs)) &&
          ok(cudaStreamWaitEvent(cout, done[l], 0))) {
        if (out_host) ok(cudaMemcpyAsync(out_host[l], out[l], q_bytes, cudaMemcpyDeviceToHost, cout));
        if (lse_host)
          ok(cudaMemcpyAsync(lse_host[l], lse[l], lse_bytes, cudaMemcpyDeviceToHost, cout));
      }
    }
    // join the copy streams back into the main stream
    if (copy_in && ok(cudaEventRecord(in_end, cin))) ok(cudaStreamWaitEvent(cs, in_end, 0));
    if (copy_out && ok(cudaEventRecord(out_end, cout))) ok(cudaStreamWaitEvent(cs, out_end, 0));
    if (cudaStreamEndCapture(cs, &graph_def) != cudaSuccess && st == PKD_OK) st = PKD_E_CUDA;
  }
  if (st == PKD_OK && cudaGraphInstantiate(&g->exec, graph_def, 0) != cudaSuccess)
    st = PKD_E_CUDA;
  if (graph_def) cudaGraphDestroy(graph_def);
  for (cudaEvent_t e : evs) cudaEventDestroy(e);
  if (cin) cudaStreamDestroy(cin);
  if (cout) cudaStreamDestroy(cout);
  if (cs) cudaStreamDestroy(cs);
  if (st != PKD_OK) {
    pkd_graph_destroy(g);
    return st;
  }
  *graph = g;
  return PKD_OK;
}

int pkd_graph_launch(pkd_graph* g, void* stream) {
  if (g == nullptr || g->exec == nullptr) return PKD_E_INVALID_ARG;
  // a dense-prefix (or cascade) graph's query maps cover the batch it was
  // captured with
  if ((g->ctx->kind.dense || g->ctx->kind.cascade) && g->ctx->info.batch != g->batch)
    return PKD_E_STALE_PLAN;
  if (cudaGraphLaunch(g->exec, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return PKD_E_CUDA;
  return PKD_OK;
}

int pkd_graph_layer_times(pkd_graph* g, float* ms) {
  if (g == nullptr || ms == nullptr || g->ev.empty()) return PKD_E_INVALID_ARG;
  for (int l = 0; l < g->layers; ++l) {
    if (cudaEventSynchronize(g->ev[2 * l + 1]) != cudaSuccess) return PKD_E_CUDA;
    if (cudaEventElapsedTime(&ms[l], g->ev[2 * l], g->ev[2 * l + 1]) != cudaSuccess)
      return PKD_E_CUDA;
  }
  return PKD_OK;
}

void pkd_graph_destroy(pkd_graph* g) {
  if (!g) return;
  if (g->exec) cudaGraphExecDestroy(g->exec);
  for (auto e : g->ev)
    if (e) cudaEventDestroy(e);
  delete g;
}

}  // extern "C"
