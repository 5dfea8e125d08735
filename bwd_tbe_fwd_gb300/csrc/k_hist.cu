// k_hist.cu -- the small-table counts x table forward path (placeholder until the tensor-core
// kernel lands: no table is routed here while histogram_supported() is false).
#include "tbe_internal.cuh"

namespace tbe {

bool histogram_supported() { return false; }

cudaError_t launch_forward_histogram(const Problem&, const tbe_tables&, const void*, const void*,
                                     const void*, float*, int, unsigned long long*,
                                     const DeviceInfo&, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace tbe
