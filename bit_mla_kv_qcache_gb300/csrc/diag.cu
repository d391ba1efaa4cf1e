// Diagnostic: a kernel whose only wait can never complete (an mbarrier that nothing arrives at),
// waited on with the bounded helper every other kernel of the library uses. The wait gives up
// after its budget and the kernel reports MLA_QCACHE_DEV_TIMEOUT in the error word and returns:
// a device-side wait ends with a status the host reads, the context stays usable.
#include "kernels.cuh"
#include "ptx.cuh"

namespace mlaq {
namespace {

__global__ void __launch_bounds__(32) wait_selftest_kernel(int32_t* err, long long budget) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  const bool ok = mbar_wait_bounded(&bar, 0, budget);  // phase 0 never completes
  if (!ok && threadIdx.x == 0) atomicOr(err, kErrTimeout);
}

}  // namespace

cudaError_t launch_wait_selftest(int32_t* err, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(err, 1ll << 21);  // ~1 ms at 2 GHz
  return cudaGetLastError();
}

}  // namespace mlaq
