// Inline-PTX building blocks shared by the sm_103a kernels of libpkd:
// mbarriers with bounded waits, TMA copies (1-D bulk and tensor-map tiles),
// proxy fences, programmatic dependent launch and the device error word.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "pkd_internal.h"

namespace pkd {
namespace dev {

constexpr unsigned kFull = 0xffffffffu;
constexpr unsigned long long kTimeoutNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity to complete.  Returns
// false on timeout, or when `abort_flag` (if given) is raised.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          const volatile int* abort_flag) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 31u) == 0) {
      if (abort_flag && *abort_flag) return false;
      if (global_ns() - t0 > kTimeoutNs) return false;
    }
  }
}

// L2 policy for the KV stream: every byte is read once per layer, so mark it
// evict-first and leave L2 to the schedule, queries and partial states.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// 1-D TMA bulk copy global -> shared, completion counted in bytes on `bar`.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// 5-D tensor-map copy global -> shared (box of the map at the given
// coordinates, innermost first), completion counted in bytes on `bar`.
__device__ __forceinline__ void tensor_copy_g2s(void* dst, const CUtensorMap* map, int c0, int c1,
                                                int c2, int c3, int c4, uint64_t* bar,
                                                uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5, %6}], [%7], %8;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4),
      "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy (TMA) writes to the same bytes.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Programmatic dependent launch: let the next kernel in the stream start its
// launch early, and wait for the previous kernel before touching its data.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void raise_error(int32_t* err, volatile int* abort_flag, int code) {
  atomicOr(err, code);
  *abort_flag = 1;
}

// Block-wide: when `want` is nonzero, thread 0 waits (bounded, kTimeoutNs)
// until the schedule header's epoch word equals it.  The plan's upload
// writes the header after the rest of the schedule, so the acquire load
// that sees the epoch also sees the whole schedule.  Every thread of the
// block must call it.  On timeout it ORs PKD_DEV_ERR_TIMEOUT into *err,
// waits for the previous grid (so that this grid's completion still implies
// the earlier ones') and returns false: the caller returns without work.
__device__ __forceinline__ bool schedule_ready(const int32_t* epoch_word_ptr, int32_t want,
                                               int32_t* err) {
  if (want == 0) return true;
  int late = 0;
  if (threadIdx.x == 0) {
    const unsigned long long t0 = global_ns();
    for (uint32_t it = 0;; ++it) {
      int32_t v;
      asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(epoch_word_ptr) : "memory");
      if (v == want) break;
      if ((it & 15u) == 15u && global_ns() - t0 > kTimeoutNs) {
        late = 1;
        break;
      }
      __nanosleep(64);
    }
  }
  if (__syncthreads_or(late)) {
    if (threadIdx.x == 0) atomicOr(err, PKD_DEV_ERR_TIMEOUT);
    pdl_wait();
    return false;
  }
  return true;
}

}  // namespace dev
}  // namespace pkd
