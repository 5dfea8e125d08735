// k_update_common.cuh -- what the classify, short-run and long-run translation units share:
// launch constants, the bucket of a width, the row-wise optimizer step on a row held by a
// group of lanes, and host-side dispatch helpers.
//
// The row-wise Adagrad rule follows "Table-Batched Embeddings in Triton", section 5: the state
// gains the mean of the squared gradient, then the row moves by lr * g / (sqrt(state) + eps).
#pragma once

#include "tbe_internal.cuh"

namespace tbe {
namespace {

constexpr unsigned FULL = 0xffffffffu;
constexpr int kThreads = 256;
constexpr int kWorkShort0 = 16;   // counters[16 + k]: work-claim counter of short bucket k
constexpr int kWorkLong = 28;     // counters[28]: work-claim counter of long chunks
constexpr int kClaim = 8;         // runs (per group) claimed per atomic in persistent mode

__device__ __forceinline__ int bucket_of_width(int D) { return D <= 1 ? 0 : 32 - __clz(D - 1); }

// ------------------------------------------------------------------------------------------
// optimizer on one row held by `nl` lanes, each lane owning float4 slices j*LPRV + li
// ------------------------------------------------------------------------------------------
template <typename WT, int OPT, typename Acc, int VPL>
__device__ __forceinline__ void apply_row_group(WT* wrow, float* state_ptr, Acc (&g)[VPL][4], int li,
                                                int lanes, int nv, int D, float lr, float eps,
                                                unsigned mask) {
  using IO = VecIO<WT, 4 * sizeof(WT)>;
  using Raw = typename IO::Raw;
  Acc scale = static_cast<Acc>(lr);
  if (OPT == TBE_OPT_ROWWISE_ADAGRAD) {
    Acc ss = 0;
#pragma unroll
    for (int j = 0; j < VPL; ++j)
      if (li + j * lanes < nv)
#pragma unroll
        for (int i = 0; i < 4; ++i) ss += g[j][i] * g[j][i];
    for (int m = lanes >> 1; m > 0; m >>= 1) ss += __shfl_xor_sync(mask, ss, m);
    const Acc s_new = static_cast<Acc>(*state_ptr) + ss / static_cast<Acc>(D);
    __syncwarp(mask);
    if (li == 0) *state_ptr = static_cast<float>(s_new);
    if constexpr (sizeof(Acc) == 8)
      scale = static_cast<Acc>(lr) / (sqrt(s_new) + static_cast<Acc>(eps));
    else
      scale = lr / (sqrtf(s_new) + eps);
  }
  Raw* wv = reinterpret_cast<Raw*>(wrow);
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    const int vec = li + j * lanes;
    if (vec < nv) {
      float f[4];
      IO::unpack(wv[vec], f);
      float o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) o[i] = static_cast<float>(static_cast<Acc>(f[i]) - scale * g[j][i]);
      wv[vec] = IO::pack(o);
    }
  }
}

// The same optimizer step for a row whose weights (raw vectors wv) and state (s_old) were
// loaded before the gradient sum.
template <typename WT, int OPT, typename Acc, int VPL>
__device__ __forceinline__ void apply_row_prefetched(
    WT* wrow, float* state_ptr, float s_old,
    const typename VecIO<WT, 4 * sizeof(WT)>::Raw (&wv)[VPL], Acc (&g)[VPL][4], int li, int lanes,
    int nv, int D, float lr, float eps, unsigned mask) {
  using IO = VecIO<WT, 4 * sizeof(WT)>;
  using Raw = typename IO::Raw;
  Acc scale = static_cast<Acc>(lr);
  if (OPT == TBE_OPT_ROWWISE_ADAGRAD) {
    Acc ss = 0;
#pragma unroll
    for (int j = 0; j < VPL; ++j)
      if (li + j * lanes < nv)
#pragma unroll
        for (int i = 0; i < 4; ++i) ss += g[j][i] * g[j][i];
    for (int m = lanes >> 1; m > 0; m >>= 1) ss += __shfl_xor_sync(mask, ss, m);
    const Acc s_new = static_cast<Acc>(s_old) + ss / static_cast<Acc>(D);
    if (li == 0) *state_ptr = static_cast<float>(s_new);
    if constexpr (sizeof(Acc) == 8)
      scale = static_cast<Acc>(lr) / (sqrt(s_new) + static_cast<Acc>(eps));
    else
      scale = lr / (sqrtf(s_new) + eps);
  }
  Raw* out = reinterpret_cast<Raw*>(wrow);
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    const int vec = li + j * lanes;
    if (vec < nv) {
      float f[4];
      IO::unpack(wv[j], f);
      float o[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) o[i] = static_cast<float>(static_cast<Acc>(f[i]) - scale * g[j][i]);
      out[vec] = IO::pack(o);
    }
  }
}

// Per-lookup factor of the backward: FAC_NONE (sum pooling, unweighted), FAC_PSW (the sorted
// per-sample weights, over L for mean pooling), FAC_INV_LEN (unweighted mean pooling: 1 / L of
// the lookup's bag, which the expand step writes once per bag into c.inv_len).
enum { FAC_NONE = 0, FAC_PSW = 1, FAC_INV_LEN = 2 };

int maxv_for(int max_D) {
  const int nv = max_D / 4;
  const int m = (nv + kWarp - 1) / kWarp;
  return m <= 1 ? 1 : (m <= 2 ? 2 : (m <= 4 ? 4 : 8));
}

template <typename F>
cudaError_t by_weight_type(int wdtype, F&& f) {
  switch (wdtype) {
    case TBE_F32: return f(float{});
    case TBE_F16: return f(__half{});
    default: return f(__nv_bfloat16{});
  }
}

}  // namespace
}  // namespace tbe
