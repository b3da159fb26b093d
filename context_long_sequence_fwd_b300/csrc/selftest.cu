// Self-test of the kernels' failure path: a bounded wait that runs out.
//
// Every barrier wait in the library's kernels gives up after a fixed time,
// records RA_ERR_TIMEOUT in the device status word and returns, so a lost
// arrival ends the kernel with an error the host reads instead of hanging
// the GPU.  This kernel exercises exactly that path without any fault: one
// thread waits on a shared-memory mbarrier that nothing ever arrives at.
#include <cuda_runtime.h>

#include "launch.h"
#include "sm103_ptx.cuh"

namespace ra {

namespace {

__global__ void __launch_bounds__(32) wait_timeout_selftest_kernel(int* status) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
    // no thread arrives: the wait ends after its time limit, having set the
    // status word, and the kernel exits normally
    mbar_wait(&bar, 0, status, nullptr);
  }
}

}  // namespace

cudaError_t launch_wait_timeout_selftest(int* status, cudaStream_t stream) {
  wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(status);
  return cudaGetLastError();
}

}  // namespace ra
