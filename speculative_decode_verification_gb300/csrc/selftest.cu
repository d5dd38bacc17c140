// selftest.cu - a kernel whose bounded waits are made to run out, so that
// tests can check that a stuck wait gives up, reports and leaves the context
// usable (no hang, no fault).
#include "common.cuh"
#include "internal.h"

namespace vk {

// Stays 0: the counter that nothing increments.
static __device__ int g_never_counted = 0;

// Warp 0 waits on a pipeline barrier that nothing arrives on, warp 1 for a
// count that nothing adds to.  Both use the waits of the verify kernels, with
// their normal limit, and record VERIFY_DEV_ETIMEOUT in *err when they give up.
__global__ void __launch_bounds__(64) stuck_wait_probe_kernel(int* err) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_w0, abort_w1;  // one abort word per wait, so that one timeout does not end the other
  if (threadIdx.x == 0) {
    abort_w0 = 0;
    abort_w1 = 0;
    mbar_init(smem_addr(&bar), 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(smem_addr(&bar), 0, &abort_w0, err);
  else if (threadIdx.x == 32) wait_count(&g_never_counted, 1, &abort_w1, err);
}

cudaError_t launch_stuck_wait_probe(int* err, cudaStream_t s) {
  stuck_wait_probe_kernel<<<1, 64, 0, s>>>(err);
  return cudaGetLastError();
}

}  // namespace vk
