// Self-test of the library's failure reporting.  Every wait in the kernels is
// bounded: when a pipeline stops (a copy that never lands, a peer role that
// stopped), the waiting thread gives up after one second, records a code in
// the device error word and the kernel returns, leaving the context usable.
// This kernel exercises exactly that path on purpose: it waits on an mbarrier
// that nothing ever arrives at.  No fault, trap or unbounded wait is involved.

#include "common.cuh"
#include "internal.h"

namespace logra {
namespace {

__global__ void wait_timeout_kernel(unsigned int* err) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bar), 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    volatile int* abort_p = &abort_flag;
    mbar_wait(smem_addr(&bar), 0, abort_p, err, kDevTimeoutSelfTest);  // gives up after the limit
  }
}

}  // namespace

logra_status launch_self_test_wait_timeout(cudaStream_t st) {
  unsigned int* err = device_error_word();
  if (!err) return LOGRA_ERR_CUDA;
  wait_timeout_kernel<<<1, 32, 0, st>>>(err);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "launch wait_timeout_kernel");
  return LOGRA_OK;
}

}  // namespace logra
