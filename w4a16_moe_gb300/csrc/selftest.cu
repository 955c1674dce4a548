// Diagnostic kernel for the failure path every bounded wait shares: one CTA
// waits, through mbar_wait_limit, on an mbarrier phase that needs one arrival
// no thread makes.  When the limit runs out the wait records B4_ERR_TIMEOUT
// and the wait site in the caller's status word and returns; the kernel then
// exits normally.  No trap, no unbounded loop.
#include <cuda_runtime.h>

#include "ptx.cuh"

namespace b4 {

constexpr uint32_t kSelfTestWaitSite = 90;

__global__ void wait_self_test_kernel(uint32_t* status, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int flag;
  if (threadIdx.x == 0) {
    status[0] = 0;
    status[1] = 0;
    flag = 0;
    mbar_init(&bar, 1);  // phase 0 completes on one arrival: none comes
    fence_mbar_init();
  }
  __syncthreads();
  const Abort ab{status, &flag};
  mbar_wait_limit(&bar, 0, ab, kSelfTestWaitSite, limit_ns);
}

cudaError_t launch_wait_self_test(uint32_t* status, unsigned long long limit_ns, cudaStream_t stream) {
  wait_self_test_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace b4
