// k_psw.cu -- gradient of the pooled output with respect to the per-sample weights.
//
// The pooled output of bag (t, b) is sum_p psw[p] * W_t[idx[p]] (over the bag length for mean
// pooling), so the gradient of a loss with upstream gradient grad_out with respect to psw[p] is
// the dot product of the bag's gradient row slice with the looked-up row:
//     grad_psw[p] = sum_d grad_out[b, col_t + d] * W_t[idx[p], d]      (/ L for mean pooling).
// "Modernizing Table Batched Embeddings with FBTriton", section 3, states that weighted tables
// scale each gradient row by its per-sample weight; this is the matching derivative for the
// per-sample weights themselves.  It reads the weights as they are, so it runs before the
// optimizer update changes them.
//
// GB300 design: one warp per (table, bag), with the forward's row split: next_pow2(D / vector)
// lanes per row, 32 / lanes rows per load step, 4 load steps in flight.  Each lane keeps its
// slice of the bag's gradient row in registers (loaded once per bag) and multiplies it into
// every looked-up row; the dot products are reduced inside each row group with xor-shuffles
// and written by the group's first lane.  Accumulation in fp32 (fp64 for fp32 tables).
#include "tbe_internal.cuh"

namespace tbe {
namespace {

constexpr unsigned FULL = 0xffffffffu;

struct PswArgs {
  const void* weights;
  const int64_t* woff;
  const int32_t* doff;
  const int64_t* roff;
  const void* indices;
  const void* offsets;
  const float* grad_out;
  float* grad_psw;
  int64_t B, TB, num_indices;
  int total_D;
  int mean;
};

__device__ __forceinline__ int pow2_at_least(int v) { return v <= 1 ? 1 : 1 << (32 - __clz(v - 1)); }

template <typename WT, typename IT, int VB, int MAXV>
__global__ void __launch_bounds__(256) psw_grad_kernel(PswArgs a) {
  using IO = VecIO<WT, VB>;
  using Raw = typename IO::Raw;
  using Acc = typename IO::Acc;
  constexpr int NE = IO::N;
  constexpr int UNROLL = MAXV >= 4 ? 1 : (MAXV == 2 ? 2 : 4);
  const int lane = lane_id();
  const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t u = warp0; u < a.TB; u += nwarps) {
    const int t = static_cast<int>(u / a.B);
    const int64_t b = u - static_cast<int64_t>(t) * a.B;
    const int col0 = __ldg(a.doff + t);
    const int D = __ldg(a.doff + t + 1) - col0;
    const int64_t E = __ldg(a.roff + t + 1) - __ldg(a.roff + t);
    const Raw* table = reinterpret_cast<const Raw*>(static_cast<const WT*>(a.weights) + __ldg(a.woff + t));
    const int nvec = D / NE;
    const int lpr = nvec >= kWarp ? kWarp : pow2_at_least(nvec);
    const int rps = kWarp / lpr;
    const int slot = lane / lpr, vi = lane & (lpr - 1);
    const int64_t s = clamp64(ld_int<IT>(a.offsets, u), 0, a.num_indices);
    const int64_t e = clamp64(ld_int<IT>(a.offsets, u + 1), s, a.num_indices);
    if (e == s) continue;  // warp-uniform
    // this lane's slice of the bag's gradient row
    Acc g[MAXV][NE];
#pragma unroll
    for (int m = 0; m < MAXV; ++m) {
      const int vv = vi + m * kWarp;
#pragma unroll
      for (int i = 0; i < NE; ++i)
        g[m][i] = vv < nvec ? static_cast<Acc>(__ldg(a.grad_out + b * a.total_D + col0 + vv * NE + i)) : Acc(0);
    }
    const Acc inv_len = a.mean ? Acc(1) / static_cast<Acc>(e - s) : Acc(1);
    for (int64_t base = s; base < e; base += kWarp) {
      const int n = static_cast<int>(min(static_cast<int64_t>(kWarp), e - base));
      int32_t my_id = -1;
      if (lane < n) {
        const int64_t v = ld_int<IT>(a.indices, base + lane);
        my_id = (v >= 0 && v < E) ? static_cast<int32_t>(v) : -1;  // E < 2^31
      }
      for (int j = 0; j < n; j += rps * UNROLL) {
        Raw v[UNROLL][MAXV];
#pragma unroll
        for (int q = 0; q < UNROLL; ++q) {
          const int r = j + q * rps + slot;
          const int32_t id = __shfl_sync(FULL, my_id, r & (kWarp - 1));
          const bool ok = r < n && id >= 0;
          const Raw* row = table + static_cast<int64_t>(ok ? id : 0) * nvec;
#pragma unroll
          for (int m = 0; m < MAXV; ++m) {
            const int vv = vi + m * kWarp;
            v[q][m] = (ok && vv < nvec) ? ldg_raw(row + vv) : Raw{};
          }
        }
#pragma unroll
        for (int q = 0; q < UNROLL; ++q) {
          Acc dot = 0;
#pragma unroll
          for (int m = 0; m < MAXV; ++m) {
            float f[NE];
            IO::unpack(v[q][m], f);
#pragma unroll
            for (int i = 0; i < NE; ++i) dot += g[m][i] * static_cast<Acc>(f[i]);
          }
          for (int off = lpr >> 1; off > 0; off >>= 1) dot += __shfl_xor_sync(FULL, dot, off);
          const int r = j + q * rps + slot;
          if (vi == 0 && r < n) a.grad_psw[base + r] = static_cast<float>(dot * inv_len);
        }
      }
    }
  }
}

template <typename WT, typename IT, int VB, int MAXV>
cudaError_t launch_psw_t(const PswArgs& a, const DeviceInfo& dev, cudaStream_t s) {
  auto k = psw_grad_kernel<WT, IT, VB, MAXV>;
  const int64_t want = (a.TB + 7) / 8;  // one bag per warp
  const int grid = persistent_grid(k, 256, 0, dev, want);
  k<<<grid, 256, 0, s>>>(a);
  note_launch();
  return cudaGetLastError();
}

template <typename WT, typename IT, int VB>
cudaError_t dispatch_psw_maxv(const PswArgs& a, int maxv, const DeviceInfo& dev, cudaStream_t s) {
  switch (maxv) {
    case 1: return launch_psw_t<WT, IT, VB, 1>(a, dev, s);
    case 2: return launch_psw_t<WT, IT, VB, 2>(a, dev, s);
    case 4: return launch_psw_t<WT, IT, VB, 4>(a, dev, s);
    default: return launch_psw_t<WT, IT, VB, 8>(a, dev, s);
  }
}

template <typename WT, typename IT>
cudaError_t dispatch_psw_vb(const PswArgs& a, int vb, int maxv, const DeviceInfo& dev, cudaStream_t s) {
  if constexpr (sizeof(WT) == 4) {
    return dispatch_psw_maxv<WT, IT, 16>(a, maxv, dev, s);
  } else {
    if (vb == 16) return dispatch_psw_maxv<WT, IT, 16>(a, maxv, dev, s);
    return dispatch_psw_maxv<WT, IT, 8>(a, maxv, dev, s);
  }
}

template <typename WT>
cudaError_t dispatch_psw_it(const PswArgs& a, int itype, int vb, int maxv, const DeviceInfo& dev, cudaStream_t s) {
  return itype == TBE_I32 ? dispatch_psw_vb<WT, int32_t>(a, vb, maxv, dev, s)
                          : dispatch_psw_vb<WT, int64_t>(a, vb, maxv, dev, s);
}

}  // namespace

cudaError_t launch_psw_gradient(const Problem& P, const tbe_tables& tab, const void* weights,
                                const void* indices, const void* offsets, const float* grad_out,
                                float* grad_psw, const DeviceInfo& dev, cudaStream_t s) {
  if (P.TB == 0 || P.num_indices == 0) return cudaSuccess;
  PswArgs a;
  a.weights = weights;
  a.woff = tab.weight_offsets;
  a.doff = tab.D_offsets;
  a.roff = tab.row_offsets;
  a.indices = indices;
  a.offsets = offsets;
  a.grad_out = grad_out;
  a.grad_psw = grad_psw;
  a.B = P.B;
  a.TB = P.TB;
  a.num_indices = P.num_indices;
  a.total_D = P.total_D;
  a.mean = P.pooling == TBE_POOL_MEAN;
  const int vb = P.vec_bytes;
  const int ne = vb / P.wbytes;
  const int max_nvec = P.max_D / ne;
  int maxv = (max_nvec + kWarp - 1) / kWarp;
  maxv = maxv <= 1 ? 1 : (maxv <= 2 ? 2 : (maxv <= 4 ? 4 : 8));
  switch (P.wdtype) {
    case TBE_F32: return dispatch_psw_it<float>(a, P.itype, vb, maxv, dev, s);
    case TBE_F16: return dispatch_psw_it<__half>(a, P.itype, vb, maxv, dev, s);
    default: return dispatch_psw_it<__nv_bfloat16>(a, P.itype, vb, maxv, dev, s);
  }
}

}  // namespace tbe
