// selftest.cu -- exercises the bounded-wait machinery every kernel relies on.
//
// One CTA initialises an mbarrier that nothing will ever arrive at and waits
// on it with the library's bounded wait.  The wait gives up after its time
// limit, the kernel reports HB_DEVERR_TIMEOUT in the device error word and
// returns normally, so the host sees HB_ERR_TIMEOUT from hb_check() and the
// CUDA context stays usable.  No fault, trap or endless loop is involved.
#include <cuda_runtime.h>

#include "hb_internal.h"
#include "ptx.cuh"

namespace hb {

__global__ void wait_timeout_kernel(int* dev_error) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  volatile int* ab = &abort_flag;
  if (threadIdx.x == 0 && !mbar_wait(&bar, 0u, ab)) report_error(dev_error, HB_DEVERR_TIMEOUT);
  __syncthreads();
}

cudaError_t launch_wait_timeout(int* dev_error, cudaStream_t stream) {
  wait_timeout_kernel<<<1, 32, 0, stream>>>(dev_error);
  return cudaGetLastError();
}

}  // namespace hb
