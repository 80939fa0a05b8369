// Self-test of the bounded device-side wait (moe_debug_wait_selftest).
//
// One warp initialises an mbarrier that expects one arrival, makes no arrival
// and issues no asynchronous copy, then waits on it with the library's bounded
// wait.  The wait must give up after `spin_limit` polls and the kernel must
// latch MOE_ERR_TIMEOUT in the status word and return, exactly as a product
// kernel does when one of its copies never lands.  Nothing is in flight when
// the kernel exits, so giving up is safe.
#include "internal.h"
#include "sm100.cuh"

namespace nvmoe {

namespace {

__global__ void wait_selftest_kernel(int* status, uint32_t spin_limit) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    sm100::mbar_init(&bar, 1);
    sm100::fence_barrier_init();
  }
  __syncthreads();
  bool ok = true;
  if (threadIdx.x == 0) ok = sm100::wait_parity_n(&bar, 0, spin_limit);
  if (!ok) latch_status(status, MOE_ERR_TIMEOUT);
}

}  // namespace

cudaError_t launch_wait_selftest(int* status, uint32_t spin_limit, cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(status, spin_limit);
  return cudaGetLastError();
}

}  // namespace nvmoe
