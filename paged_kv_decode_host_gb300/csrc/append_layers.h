// The every-layer form of the append (append_kernel.cu): one launch writes a
// step's new K / V rows into every layer's cache.
#pragma once

#include <stdint.h>

#include <cuda_runtime_api.h>

namespace pkd {

// Per-layer pointers, passed to the kernel as one argument block.
constexpr int kMaxAppendLayers = 128;
struct AppendLayers {
  const void* k_new[kMaxAppendLayers];
  const void* v_new[kMaxAppendLayers];
  void* kv[kMaxAppendLayers];
};

cudaError_t launch_append_layers(const AppendLayers& L, int32_t layers,
                                 const int32_t* batch_indices, const int32_t* positions,
                                 int32_t n, const int32_t* indptr, const int32_t* indices,
                                 const int32_t* last_page_len, int32_t batch, int32_t num_pages,
                                 int32_t page_size, int32_t hkv, int32_t head_bytes, bool hnd,
                                 int32_t* err, cudaStream_t stream);

}  // namespace pkd
