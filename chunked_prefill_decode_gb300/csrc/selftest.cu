// selftest.cu -- exercises the bounded-wait machinery every kernel relies on.
//
// One CTA initialises an mbarrier that nothing will ever arrive at and waits
// on it with the library's bounded wait.  The wait gives up after its time
// limit, the kernel reports HB_DEVERR_TIMEOUT in the device error word and
// returns normally, so the host sees HB_ERR_TIMEOUT from hb_check() and the
// CUDA context stays usable.  No fault, trap or endless loop is involved.
// The second test does the same with the flag wait of hb_step's append.
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

// A device word that nothing raises: the flag of flag_timeout_kernel.
__device__ uint32_t g_flag_never_raised = 0;

// The wait hb_step's append kernel does on its slot's flag (warp_wait_flag),
// on a flag that stays 0: every warp gives up after the time limit and the
// kernel reports HB_DEVERR_TIMEOUT.
__global__ void flag_timeout_kernel(int* dev_error) {
  if (!__syncthreads_and(warp_wait_flag(&g_flag_never_raised, 1u, dev_error))) return;
}

cudaError_t launch_flag_timeout(int* dev_error, cudaStream_t stream) {
  flag_timeout_kernel<<<1, 64, 0, stream>>>(dev_error);
  return cudaGetLastError();
}

}  // namespace hb
