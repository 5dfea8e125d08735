// tbe_noalloc.cu -- tbe_backward_update_noalloc: the backward update for callers that cannot
// allocate device memory.
//
// Some callers have no way to hand the library a workspace: code running where every device
// allocation must be planned ahead of time (a fixed memory budget, a custom allocator that
// cannot be reached from the calling layer, an embedded runtime with cudaMalloc forbidden after
// start-up).  This entry point runs the same backward as tbe_backward_update, but its scratch
// memory is a fixed-size array compiled into the library instead of a caller-provided buffer.
//
// The array lives in device global memory from the time the library's module is loaded on a
// device until the process exits: with lazy module loading (CUDA's default) that is the first use
// of the library on that device, with CUDA_MODULE_LOADING=EAGER every device whose context loads
// the library, whether or not this entry point is ever called there.  Host code only ever sees a
// host-side stand-in for its name; the real device address is looked up once per device with
// cudaGetSymbolAddress (with that device current) during the first call on that device, so that
// first call should be made before any stream capture.  The address is kept for the life of the
// process: after a cudaDeviceReset (which ends the context the address belongs to) the library
// must be loaded again before this entry point is used on that device.  All calls on a device share the one array: calls whose
// work overlaps on the GPU (different streams without ordering, or different host threads)
// race on it and must be serialized by the caller.  The backward itself zeroes the counters it
// needs at the start of every call and writes every other scratch byte before reading it, so
// the previous call's leftovers never matter.
#include <mutex>

#include "tbe_internal.cuh"

namespace {

// Scratch for one backward update; problems whose backward workspace is larger are rejected.
static __device__ __align__(256) unsigned char g_tbe_static_scratch[TBE_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device (looked up once per device).
cudaError_t scratch_on_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_tbe_static_scratch);
    if (e != cudaSuccess) return e;
    if (p == nullptr) return cudaErrorInvalidSymbol;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" {

tbe_status tbe_backward_update_noalloc(const tbe_problem* prob, const tbe_options* opt,
                                       const tbe_tables* tables, void* weights, float* state,
                                       const void* indices, const void* offsets, const float* psw,
                                       const float* grad_out, tbe_optimizer optimizer, float lr,
                                       float eps, int64_t* d_stats, void* stream) {
  if (opt != nullptr && opt->prepared) return TBE_ERR_INVALID_ARG;  // nothing prepares the built-in array
  const size_t need = tbe_backward_workspace_size(prob, opt);
  if (need == 0) {
    // the problem or the options were rejected: the workspace entry point's argument checks
    // (which run before any launch) give the status it would return
    return tbe_backward_update(prob, opt, tables, weights, state, indices, offsets, psw, grad_out, optimizer,
                               lr, eps, nullptr, 0, d_stats, stream);
  }
  if (need > TBE_STATIC_SCRATCH_BYTES) return TBE_ERR_WORKSPACE;
  void* scratch = nullptr;
  const cudaError_t e = scratch_on_current_device(&scratch);
  if (e != cudaSuccess) return tbe::cuda_status(e);  // recorded for tbe_last_cuda_error
  return tbe_backward_update(prob, opt, tables, weights, state, indices, offsets, psw, grad_out,
                             optimizer, lr, eps, scratch, TBE_STATIC_SCRATCH_BYTES, d_stats, stream);
}

}  // extern "C"
