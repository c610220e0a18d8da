// append_paged_kv_cache for sm_103a: write new tokens' K and V rows into
// their page slots (pyshine FlashInfer tour, "The Paged KV Cache Layer": the
// engine calls it after every generated token; rows are copied into page
// slots, a token's page found through the page table).
//
// Token i belongs to request b = batch_indices[i] at position pos =
// positions[i] (0-based within the request's length after the append); its
// K row goes to cache[indices[indptr[b] + pos / P]][0][pos % P][:][:] and its
// V row to [...][1][pos % P][:][:] (NHD, FlashInfer, in depth, "The
// block-sparse page table"); in the HND layout head h's part goes to
// [page][0 or 1][h][pos % P][:] ("FlashInfer 完全拆解", 接口层最容易踩的四个坑).
// One warp per token (and layer, for the every-layer form), 16-byte vector
// copies; the table is read on the device.
// Elements are moved as bytes (bf16 or e4m3 alike).  A token whose request,
// position or page id falls outside the table is skipped and flagged in the
// error word -- the kernel never writes outside the cache.
#include <cuda_runtime.h>
#include <stdint.h>

#include "append_layers.h"
#include "pkd_internal.h"

namespace pkd {
namespace {

constexpr int kAppendWarps = 8;

// Page and slot of token i (lane 0 looks them up, the warp shares them), or
// page -1 when the token falls outside the table (flagged in the error word).
__device__ __forceinline__ void token_slot(int64_t i, const int32_t* __restrict__ batch_indices,
                                           const int32_t* __restrict__ positions,
                                           const int32_t* __restrict__ indptr,
                                           const int32_t* __restrict__ indices,
                                           const int32_t* __restrict__ last_page_len,
                                           int32_t batch, int32_t num_pages, int32_t page_size,
                                           int32_t* err, int lane, int& page, int& slot) {
  page = -1;
  slot = 0;
  if (lane == 0) {
    const int b = batch_indices[i];
    const int pos = positions[i];
    if (b >= 0 && b < batch) {
      const int p0 = indptr[b], p1 = indptr[b + 1];
      const int last = last_page_len[b];
      const int64_t len = (int64_t)page_size * (p1 - p0 - 1) + last;
      if (p1 > p0 && last >= 1 && last <= page_size && pos >= 0 && pos < len) {
        const int pg = indices[p0 + pos / page_size];
        if (pg >= 0 && pg < num_pages) {
          page = pg;
          slot = pos % page_size;
        }
      }
    }
    if (page < 0 && err != nullptr) atomicOr(err, PKD_DEV_ERR_BOUNDS);
  }
  page = __shfl_sync(0xffffffffu, page, 0);
  slot = __shfl_sync(0xffffffffu, slot, 0);
}

// Copy token i's K and V rows (hkv * head_chunks 16-byte chunks each) into
// slot `slot` of page `page`.
__device__ __forceinline__ void copy_rows(const uint4* __restrict__ k_new,
                                          const uint4* __restrict__ v_new,
                                          uint4* __restrict__ kv, int64_t i, int page, int slot,
                                          int32_t page_size, int32_t hkv, int32_t head_chunks,
                                          int32_t hnd, int lane) {
  // a token row is hkv * head_chunks chunks; one K (or V) page block is
  // page_size rows
  const int64_t row_chunks = (int64_t)hkv * head_chunks;
  const int64_t kv_block = (int64_t)page_size * row_chunks;    // K -> V
  const int64_t page_base = (int64_t)page * 2 * kv_block;
  const uint4* ks = k_new + i * row_chunks;
  const uint4* vs = v_new + i * row_chunks;
  for (int c = lane; c < row_chunks; c += 32) {
    int64_t dst;
    if (hnd) {
      const int h = c / head_chunks, cc = c % head_chunks;
      dst = page_base + ((int64_t)h * page_size + slot) * head_chunks + cc;
    } else {
      dst = page_base + (int64_t)slot * row_chunks + c;
    }
    kv[dst] = ks[c];
    kv[dst + kv_block] = vs[c];
  }
}

__global__ void __launch_bounds__(kAppendWarps * 32) append_kernel(
    const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
    const int32_t* __restrict__ batch_indices, const int32_t* __restrict__ positions, int32_t n,
    const int32_t* __restrict__ indptr, const int32_t* __restrict__ indices,
    const int32_t* __restrict__ last_page_len, int32_t batch, uint4* __restrict__ kv,
    int32_t num_pages, int32_t page_size, int32_t hkv, int32_t head_chunks, int32_t hnd,
    int32_t* err) {
  const int lane = threadIdx.x & 31;
  const int64_t i = (int64_t)blockIdx.x * kAppendWarps + (threadIdx.x >> 5);
  if (i >= n) return;
  int page, slot;
  token_slot(i, batch_indices, positions, indptr, indices, last_page_len, batch, num_pages,
             page_size, err, lane, page, slot);
  if (page < 0) return;
  copy_rows(k_new, v_new, kv, i, page, slot, page_size, hkv, head_chunks, hnd, lane);
}

// Every layer of a step at once: the layers share the step's table, so one
// launch covers tokens x layers (grid y = layer) instead of one launch per
// layer; the error bit is raised once, by layer 0's warps.
__global__ void __launch_bounds__(kAppendWarps * 32) append_layers_kernel(
    const __grid_constant__ AppendLayers L, const int32_t* __restrict__ batch_indices,
    const int32_t* __restrict__ positions, int32_t n, const int32_t* __restrict__ indptr,
    const int32_t* __restrict__ indices, const int32_t* __restrict__ last_page_len,
    int32_t batch, int32_t num_pages, int32_t page_size, int32_t hkv, int32_t head_chunks,
    int32_t hnd, int32_t* err) {
  const int lane = threadIdx.x & 31;
  const int64_t i = (int64_t)blockIdx.x * kAppendWarps + (threadIdx.x >> 5);
  const int layer = blockIdx.y;
  if (i >= n) return;
  int page, slot;
  token_slot(i, batch_indices, positions, indptr, indices, last_page_len, batch, num_pages,
             page_size, layer == 0 ? err : nullptr, lane, page, slot);
  if (page < 0) return;
  copy_rows(static_cast<const uint4*>(L.k_new[layer]), static_cast<const uint4*>(L.v_new[layer]),
            static_cast<uint4*>(L.kv[layer]), i, page, slot, page_size, hkv, head_chunks, hnd,
            lane);
}

}  // namespace

cudaError_t launch_append(const void* k_new, const void* v_new, const int32_t* batch_indices,
                          const int32_t* positions, int32_t n, const int32_t* indptr,
                          const int32_t* indices, const int32_t* last_page_len, int32_t batch,
                          void* kv, int32_t num_pages, int32_t page_size, int32_t hkv,
                          int32_t head_bytes, bool hnd, int32_t* err, cudaStream_t stream) {
  const int64_t blocks = ((int64_t)n + kAppendWarps - 1) / kAppendWarps;
  append_kernel<<<(unsigned)blocks, kAppendWarps * 32, 0, stream>>>(
      static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), batch_indices,
      positions, n, indptr, indices, last_page_len, batch, static_cast<uint4*>(kv), num_pages,
      page_size, hkv, head_bytes / 16, hnd ? 1 : 0, err);
  return cudaGetLastError();
}

cudaError_t launch_append_layers(const AppendLayers& L, int32_t layers,
                                 const int32_t* batch_indices, const int32_t* positions,
                                 int32_t n, const int32_t* indptr, const int32_t* indices,
                                 const int32_t* last_page_len, int32_t batch, int32_t num_pages,
                                 int32_t page_size, int32_t hkv, int32_t head_bytes, bool hnd,
                                 int32_t* err, cudaStream_t stream) {
  const int64_t blocks = ((int64_t)n + kAppendWarps - 1) / kAppendWarps;
  append_layers_kernel<<<dim3((unsigned)blocks, (unsigned)layers), kAppendWarps * 32, 0, stream>>>(
      L, batch_indices, positions, n, indptr, indices, last_page_len, batch, num_pages, page_size,
      hkv, head_bytes / 16, hnd ? 1 : 0, err);
  return cudaGetLastError();
}

}  // namespace pkd
