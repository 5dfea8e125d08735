// k_selftest.cu -- tbe_selftest_wait_timeout: drives the library's bounded mbarrier wait to its
// limit, so that the give-up path (count TBE_STAT_WAIT_TIMEOUT, return) is exercised on a GPU.
// The barrier is initialised for one arrival that never comes; nothing else is in flight, so the
// CTA can return as soon as the wait gives up.
#include "tbe_internal.cuh"
#include "tbe_selftest.h"

namespace tbe {
namespace {

__global__ void wait_timeout_kernel(uint32_t polls, unsigned long long* stats) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait_bounded(&bar, 0, polls)) stat_add(stats, TBE_STAT_WAIT_TIMEOUT, 1);
}

}  // namespace
}  // namespace tbe

extern "C" tbe_status tbe_selftest_wait_timeout(uint32_t polls, int64_t* d_stats, void* stream) {
  if (d_stats == nullptr || (reinterpret_cast<uintptr_t>(d_stats) & 7) != 0 || polls < 1 || polls > 4096)
    return TBE_ERR_INVALID_ARG;
  tbe::wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      polls, reinterpret_cast<unsigned long long*>(d_stats));
  return tbe::cuda_status(cudaGetLastError());
}
