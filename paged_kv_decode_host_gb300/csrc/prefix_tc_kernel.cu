// Dense shared-prefix kernel for sm_103a: the standalone launch of the dense
// role (prefix_tc_body.cuh, which holds the design and the device code) for
// plans made with PKD_FLAG_DENSE_PREFIX.  One CTA per SM, 384 threads.
#include <cuda_runtime.h>
#include <stdint.h>

#include "prefix_tc_body.cuh"

namespace pkd {
namespace {

__global__ void __launch_bounds__(tc::kTcThreads, 1)
    prefix_tc_kernel(const __grid_constant__ DecodeArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if (!dev::schedule_ready(a.sched + H_EPOCH, a.wait_epoch, a.err)) return;
  tc::prefix_tc_body(a, smem_raw);
}

}  // namespace

const void* prefix_tc_kernel_ptr() { return reinterpret_cast<const void*>(&prefix_tc_kernel); }

int prefix_tc_smem_bytes() { return tc::smem_bytes(); }

int prefix_tc_threads() { return tc::kTcThreads; }

}  // namespace pkd
