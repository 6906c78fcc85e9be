// Self-test of the bounded-wait path every kernel relies on: a one-CTA kernel
// waits on an mbarrier that nothing ever arrives at, with a short limit, and
// must come back with the timeout recorded in its status word instead of
// hanging.  Used by the failure-detection test; it faults nothing and leaves
// the context usable.
#include <cuda_runtime.h>

#include "fa2.h"
#include "ptx.cuh"

namespace fa2 {
namespace {

__device__ int g_selftest_status;

__global__ void wait_timeout_kernel(unsigned long long timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);  // expects one arrival that never comes
    fence_mbar_init();
  }
  __syncthreads();
  mbar_wait(&bar, 0, &g_selftest_status, timeout_ns);
}

}  // namespace
}  // namespace fa2

extern "C" int fa2_check_wait_timeout(int timeout_us, int* status_out) {
  if (!status_out) return FA2_ERR_NULL;
  if (timeout_us < 1 || timeout_us > 5000000) return FA2_ERR_SHAPE;
  const int zero = 0;
  if (cudaMemcpyToSymbol(fa2::g_selftest_status, &zero, sizeof(int)) != cudaSuccess) return FA2_ERR_CUDA;
  fa2::wait_timeout_kernel<<<1, 32>>>(static_cast<unsigned long long>(timeout_us) * 1000ull);
  if (cudaGetLastError() != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) return FA2_ERR_CUDA;
  if (cudaMemcpyFromSymbol(status_out, fa2::g_selftest_status, sizeof(int)) != cudaSuccess) return FA2_ERR_CUDA;
  return FA2_OK;
}
