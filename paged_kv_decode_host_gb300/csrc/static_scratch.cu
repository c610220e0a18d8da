// Allocation-free decode entry point: pkd_run_static_scratch.
//
// Who needs it: callers that may not call cudaMalloc (or any allocator) at
// the point where they run attention -- e.g. an engine whose memory manager
// owns every byte of device memory and forbids libraries from allocating, a
// process under a hard memory budget, or a plugin loaded into a host
// framework that gives it no allocator.  Such a caller cannot hand the
// regular path its workspace buffer (nor the pinned staging pkd_create makes).
//
// What it does instead: the schedule and the split-KV partial states live in
// one file-scope device array of fixed size, kStaticScratchBytes, which every
// GPU that loads this library keeps until the process exits.  The caller
// passes only inputs and outputs: a schedule already built on the host by
// pkd_plan_host (caller-owned host memory), q, the KV cache, out and lse.
// The entry point copies the schedule into the array, clears the device
// error word, and launches the same decode and merge kernels as pkd_run.
//
// Sharing: every call, from any thread or stream, uses the same array, which
// keeps the previous call's contents.  Calls whose work overlaps on the GPU
// race on it; callers must serialise them (one stream, or events).
//
// Set-up: the first call on each device (made with that device current)
// looks up the array's device address with cudaGetSymbolAddress and sets the
// decode kernel's shared-memory attribute.  Make that first call before any
// stream capture.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <mutex>

#include "pkd_internal.h"

namespace pkd {
namespace {

constexpr size_t kStaticScratchBytes = (size_t)32 << 20;  // 32 MiB per device
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

struct DeviceSlot {
  std::atomic<int> ready{0};
  uint8_t* addr = nullptr;
};
DeviceSlot g_slots[kMaxDevices];
std::mutex g_setup_mu;

// Device address of the scratch array on the current device (set-up once).
int scratch_address(int group, bool mma, uint8_t** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKD_E_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return PKD_E_UNSUPPORTED_SHAPE;
  DeviceSlot& s = g_slots[dev];
  const int bit = 1 << (2 * group + (mma ? 1 : 0));
  if (s.ready.load(std::memory_order_acquire) & bit) {
    *out = s.addr;
    return PKD_OK;
  }
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (s.addr == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr)
      return PKD_E_CUDA;
    s.addr = static_cast<uint8_t*>(p);
  }
  DecodeKind k;
  k.group = group;
  k.mma = mma;
  if (decode_prepare(k, decode_smem_bytes(kMaxKvHeads, k)) != cudaSuccess) return PKD_E_CUDA;
  s.ready.fetch_or(bit, std::memory_order_release);
  *out = s.addr;
  return PKD_OK;
}

// A schedule handed in from the host is checked before it reaches the GPU:
// it must have been planned for this very layout (same capacities, hence the
// same word offsets), and every index the kernels follow from it must stay
// inside the arrays and the scratch: CTA queues monotone within the item
// list, each item's requests inside the batch, its pages inside the page
// list and its partial-state slots below the layout's slot count; each split
// request's slots likewise.  O(items + units) on the host.
bool schedule_fits(const int32_t* w, const Layout& L) {
  const int32_t batch = w[H_BATCH], n_cta = w[H_NCTA], n_items = w[H_NITEMS];
  const int32_t n_units = w[H_NUNITS], nnz = w[H_NNZ], P = w[H_P];
  if (batch < 0 || n_units < 0 || n_units > L.max_items || P < 1) return false;
  const int32_t* cta = w + L.cta_indptr;
  if (cta[0] != 0 || cta[n_cta] != n_items) return false;
  for (int32_t c = 0; c < n_cta; ++c)
    if (cta[c + 1] < cta[c]) return false;
  for (int32_t j = 0; j < n_items; ++j) {
    const int32_t* it = w + L.items + (int64_t)j * kItemWords;
    const int32_t req = it[0], t0 = it[1], t1 = it[2], slot = it[3], page0 = it[4];
    const int32_t n_req = it[5], stride = it[6];
    if (n_req != 1 || req < 0 || req >= batch || t0 < 0 || t1 <= t0) return false;
    if (page0 < 0 || (int64_t)page0 + (t1 - 1 - t0 + (t0 % P)) / P >= nnz) return false;
    if (slot < -1 || slot >= L.max_slots || stride < 0) return false;
  }
  const int32_t* units = w + L.units;
  const int32_t* merge = w + L.merge_indptr;
  if (merge[0] != 0) return false;
  for (int32_t u = 0; u < n_units; ++u)
    if (units[2 * u] < 0 || units[2 * u] >= batch || merge[u + 1] < merge[u] ||
        merge[u + 1] > L.max_slots)
      return false;
  return true;
}

// The configuration checks shared by both entry points of this file.
int check_static_config(const pkd_config* cfg, int* group) {
  if (cfg == nullptr) return PKD_E_INVALID_ARG;
  if ((cfg->flags & ~(PKD_FLAG_FMA_CONSUMER | PKD_FLAG_MMA_CONSUMER)) != 0 ||
      cfg->flags == (PKD_FLAG_FMA_CONSUMER | PKD_FLAG_MMA_CONSUMER) || cfg->num_ctas < 1 ||
      cfg->head_dim != kHeadDim || cfg->num_kv_heads < 1 || cfg->num_kv_heads > kMaxKvHeads ||
      cfg->num_qo_heads < 1 || cfg->num_qo_heads % cfg->num_kv_heads != 0 ||
      cfg->page_size < 1 || cfg->num_pages < 1 || cfg->max_batch < 0 || cfg->max_num_pages < 0)
    return PKD_E_INVALID_ARG;
  *group = cfg->num_qo_heads / cfg->num_kv_heads;
  if (*group != 1 && *group != 2 && *group != 4 && *group != 8) return PKD_E_UNSUPPORTED_SHAPE;
  if (make_layout(*cfg, cfg->num_ctas).total_bytes > kStaticScratchBytes)
    return PKD_E_SCRATCH_LIMIT;
  return PKD_OK;
}

}  // namespace
}  // namespace pkd

using namespace pkd;

extern "C" int pkd_run_static_scratch(const pkd_config* cfg, const int32_t* schedule_words,
                                      size_t num_words, const void* q, const void* kv, void* out,
                                      float* lse, void* stream) {
  int group = 0;
  int st = check_static_config(cfg, &group);
  if (st != PKD_OK) return st;
  if (schedule_words == nullptr) return PKD_E_INVALID_ARG;
  const Layout L = make_layout(*cfg, cfg->num_ctas);
  // the schedule must be pkd_plan_host's output for this very configuration
  if ((int64_t)num_words < L.page_list) return PKD_E_INVALID_ARG;
  const int32_t* h = schedule_words;
  if (h[H_MAGIC] != kMagic || h[H_HQ] != cfg->num_qo_heads || h[H_HKV] != cfg->num_kv_heads ||
      h[H_D] != cfg->head_dim || h[H_P] != cfg->page_size || h[H_NCTA] != cfg->num_ctas ||
      h[H_MAXBATCH] != cfg->max_batch || h[H_MAXPAGES] != cfg->max_num_pages ||
      h[H_BATCH] < 0 || h[H_BATCH] > cfg->max_batch || h[H_BLOCK] != 1 ||
      h[H_NITEMS] < 0 || h[H_NITEMS] > L.max_items || h[H_NNZ] < 0 ||
      h[H_NNZ] > cfg->max_num_pages || (int64_t)num_words < L.page_list + h[H_NNZ] ||
      !schedule_fits(h, L))
    return PKD_E_INVALID_ARG;
  if (h[H_BATCH] > 0) {
    if (q == nullptr || kv == nullptr || out == nullptr) return PKD_E_INVALID_ARG;
    if (((uintptr_t)q | (uintptr_t)kv | (uintptr_t)out) % 16 != 0 || (uintptr_t)lse % 4 != 0)
      return PKD_E_INVALID_ARG;
  }
  const bool mma = use_mma_consumer(group, cfg->flags);
  uint8_t* ws = nullptr;
  st = scratch_address(group, mma, &ws);
  if (st != PKD_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t sched_bytes = ((size_t)L.page_list + (size_t)h[H_NNZ]) * 4;
  if (cudaMemcpyAsync(ws, schedule_words, sched_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return PKD_E_CUDA;
  if (cudaMemsetAsync(ws + L.err_byte, 0, 4, s) != cudaSuccess) return PKD_E_CUDA;

  DecodeArgs a{};
  a.sched = reinterpret_cast<const int32_t*>(ws);
  a.o_part = reinterpret_cast<float*>(ws + L.o_part_byte);
  a.l_part = reinterpret_cast<float*>(ws + L.l_part_byte);
  a.err = reinterpret_cast<int32_t*>(ws + L.err_byte);
  a.q = static_cast<const uint16_t*>(q);
  a.kv = static_cast<const uint8_t*>(kv);
  a.out = static_cast<uint16_t*>(out);
  a.lse = lse;
  a.row_bytes = cfg->num_kv_heads * kHeadDim * 2;
  a.page_bytes = (int64_t)2 * cfg->page_size * a.row_bytes;
  a.off_cta = L.cta_indptr;
  a.off_items = L.items;
  a.off_pages = L.page_list;
  a.hq = cfg->num_qo_heads;
  a.hkv = cfg->num_kv_heads;
  a.page_size = cfg->page_size;
  a.num_pages = cfg->num_pages;
  a.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)cfg->head_dim));
  a.v_scale = 1.f;
  DecodeKind k;   // token-row producer
  k.group = group;
  k.mma = mma;
  if (launch_decode(k, a, cfg->num_ctas, cfg->num_kv_heads, decode_smem_bytes(cfg->num_kv_heads, k),
                    s) != cudaSuccess)
    return PKD_E_CUDA;
  MergeArgs m{};
  m.sched = a.sched;
  m.o_part = a.o_part;
  m.l_part = a.l_part;
  m.out = a.out;
  m.lse = lse;
  m.off_units = L.units;
  m.off_merge = L.merge_indptr;
  m.hq = cfg->num_qo_heads;
  if (launch_merge_partials(m, merge_grid_for(cfg->num_ctas), h[H_MAXCHUNKS], s) != cudaSuccess)
    return PKD_E_CUDA;
  return PKD_OK;
}

extern "C" int pkd_static_scratch_last_error(const pkd_config* cfg, void* stream,
                                             int32_t* dev_err) {
  int group = 0;
  int st = check_static_config(cfg, &group);
  if (st != PKD_OK) return st;
  if (dev_err == nullptr) return PKD_E_INVALID_ARG;
  uint8_t* ws = nullptr;
  st = scratch_address(group, use_mma_consumer(group, cfg->flags), &ws);
  if (st != PKD_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t off = make_layout(*cfg, cfg->num_ctas).err_byte;
  int32_t v = 0;
  // stream-ordered read of the word, then its reset, then a wait for this
  // stream only (pageable destination: the copy completes before it returns)
  if (cudaMemcpyFromSymbolAsync(&v, g_static_scratch, sizeof v, off, cudaMemcpyDeviceToHost, s) !=
      cudaSuccess)
    return PKD_E_CUDA;
  if (cudaMemsetAsync(ws + off, 0, sizeof v, s) != cudaSuccess) return PKD_E_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return PKD_E_CUDA;
  *dev_err = v;
  return PKD_OK;
}
