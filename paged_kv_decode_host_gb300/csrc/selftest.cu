// Self-test of the kernels' bounded waits (failure detection without a GPU
// fault): one CTA of two warps whose waits, on shared-memory mbarriers that
// nothing ever arrives on, go through the same dev::mbar_wait the decode and
// prefix kernels use.
//  * warp 0 waits with no abort flag: the wait gives up after the kernels'
//    limit (kTimeoutNs), then raises PKD_DEV_ERR_TIMEOUT and the CTA's abort
//    flag, as a kernel role does when its input never lands;
//  * warp 1 (mode 1) starts its own wait half a limit later, with the abort
//    flag: it has to return as soon as warp 0 raises the flag, before its own
//    limit -- the path by which the other roles of a kernel stop.
// Each wait's duration goes to wait_ns[0..1].  The kernel ends after about one
// wait limit; it issues no copy and no tensor-core work, so nothing is left
// in flight.
#include <cuda_runtime.h>
#include <stdint.h>

#include "pkd_internal.h"
#include "sm103_ptx.cuh"

namespace pkd {
namespace {

using namespace dev;

__global__ void __launch_bounds__(64, 1)
    bounded_wait_selftest(int mode, int32_t* err, unsigned long long* wait_ns) {
  __shared__ uint64_t bar[2];
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  volatile int* abort = &abort_flag;
  if (warp == 0) {
    const unsigned long long t0 = global_ns();
    const bool ok = mbar_wait(&bar[0], 0, nullptr);
    const unsigned long long t1 = global_ns();
    if (!__all_sync(kFull, ok) && lane == 0) raise_error(err, abort, PKD_DEV_ERR_TIMEOUT);
    if (lane == 0) wait_ns[0] = t1 - t0;
  } else if (mode == 1) {
    // half a limit late: the peer's limit ends first, its flag must end this wait
    const unsigned long long start = global_ns();
    while (global_ns() - start < kTimeoutNs / 2) {
    }
    const unsigned long long t0 = global_ns();
    const bool ok = mbar_wait(&bar[1], 0, abort);
    const unsigned long long t1 = global_ns();
    if (lane == 0) wait_ns[1] = ok ? 0ull : t1 - t0;
  } else if (lane == 0) {
    wait_ns[1] = 0;
  }
}

}  // namespace
}  // namespace pkd

extern "C" int pkd_selftest_bounded_wait(int32_t mode, int32_t* d_err,
                                         unsigned long long* d_wait_ns, void* stream) {
  if ((mode != 0 && mode != 1) || d_err == nullptr || d_wait_ns == nullptr)
    return PKD_E_INVALID_ARG;
  pkd::bounded_wait_selftest<<<1, 64, 0, static_cast<cudaStream_t>(stream)>>>(mode, d_err,
                                                                             d_wait_ns);
  return cudaGetLastError() == cudaSuccess ? PKD_OK : PKD_E_CUDA;
}
