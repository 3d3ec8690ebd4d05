// Self-test of the device-side failure path: every mbarrier wait of the
// kernels is bounded, and on expiry raises kStatusWaitTimeout in the status
// word and returns instead of hanging the GPU.  This kernel waits on a
// barrier that no thread and no copy completes, so the bound expires (about
// 2 s), and the host can check the status word and that the context still
// works afterwards.
#include <stdint.h>

#include "async_copy.cuh"
#include "orca_internal.h"

namespace orca {
namespace {

__global__ void wait_selftest_kernel(int32_t *status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();
  // phase 0 never completes: its one expected arrival never comes
  if (threadIdx.x == 0) mbar_wait(&bar, 0, &abort_flag, status);
  __syncthreads();
}

}  // namespace

cudaError_t launch_wait_selftest(int32_t *status, cudaStream_t st) {
  wait_selftest_kernel<<<1, 32, 0, st>>>(status);
  return cudaGetLastError();
}

}  // namespace orca
