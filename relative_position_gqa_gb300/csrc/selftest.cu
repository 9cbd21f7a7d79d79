// Self-test of the bounded waits that every pipeline kernel relies on.  One thread per
// CTA waits, with the kernels' own mbar_wait, on an mbarrier that nothing will ever arrive
// on: the wait must give up by itself (after its cycle budget, about two seconds) and the
// kernel must report INKLING_ERR_TIMEOUT and return, leaving the context usable.  In the
// second mode CTA 0 reports an error first, and the waits of the other CTAs must notice
// the launch's status word and give up early instead of running out their budget.  No
// fault, trap or unbounded wait is involved.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/inkling.h"
#include "ptx.cuh"

namespace ink {

__global__ void __launch_bounds__(32) wait_selftest_kernel(int mode, int* status, int* gave_up) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x != 0) return;
  if (mode == 1 && blockIdx.x == 0) {
    report(status, kErrBadInput);  // "another CTA already failed"
    return;
  }
  if (!mbar_wait(&bar, 0, &abort_flag, status)) {  // nothing arrives: phase 0 never completes
    report(status, kErrTimeout);
    atomicAdd(gave_up, 1);
  }
}

}  // namespace ink

extern "C" int inkling_selftest_bounded_wait(int32_t mode, int32_t ctas, int32_t* dev_status,
                                             int32_t* dev_gave_up, inkling_stream_t stream) {
  if ((mode != 0 && mode != 1) || ctas < 1 || ctas > 1024 || !dev_status || !dev_gave_up)
    return INKLING_ERR_INVALID_ARG;
  ink::wait_selftest_kernel<<<ctas, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      mode, dev_status, dev_gave_up);
  return cudaGetLastError() == cudaSuccess ? INKLING_OK : INKLING_ERR_CUDA;
}
