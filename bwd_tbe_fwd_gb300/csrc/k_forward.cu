// k_forward.cu -- pooled forward gather.
//
// "Modernizing Table Batched Embeddings with FBTriton", section 2 ("The general gather
// path"): for each table and bag, gather the indexed rows, optionally scale them by the
// per-sample weight, accumulate in fp32 (fp64 for fp32 tables) and write one D-wide pooled
// output row.  The pages' design is a Triton program per group of bags looping over the tables
// with four to eight row loads in flight; here the unit of work is one (table, bag) per warp:
//   * the warp reads up to 32 ids of its bag with one coalesced load and broadcasts them with
//     shuffles (the id -> row dependence is the latency to hide);
//   * a row of D elements is split into 16-byte vectors; a group of next_pow2(vectors) lanes
//     covers one row, so one warp-wide load instruction fetches 32/group rows, and UNROLL such
//     instructions are issued before any is consumed (8 rows in flight per warp for fp16 D=128);
//   * the row groups are reduced with xor-shuffles and one group writes the fp32 result with
//     streaming 16-byte stores;
//   * warps walk the (table, bag) units table-major with a grid stride, so the offsets and ids a
//     CTA reads are contiguous and every warp of a CTA usually sees the same D.
// Out-of-range ids are repaired to row 0 in flight when fused bounds checking is on (writing
// the repaired id back), else skipped and counted; no id outside its table is dereferenced.
#include "tbe_internal.cuh"

namespace tbe {
namespace {

struct FwdArgs {
  const void* weights;
  const int64_t* woff;
  const int32_t* doff;
  const int64_t* roff;
  void* indices;
  const void* offsets;
  const float* psw;
  float* out;
  int64_t B;
  int64_t num_indices;
  int64_t unit_begin, unit_end;
  int total_D;
  int fused_bounds;
  unsigned long long* stats;
};

__device__ __forceinline__ int next_pow2_int(int v) { return v <= 1 ? 1 : 1 << (32 - __clz(v - 1)); }

__device__ __forceinline__ void store_out(float* dst, const float (&v)[8]) {
  __stcs(reinterpret_cast<float4*>(dst), make_float4(v[0], v[1], v[2], v[3]));
  __stcs(reinterpret_cast<float4*>(dst) + 1, make_float4(v[4], v[5], v[6], v[7]));
}
__device__ __forceinline__ void store_out(float* dst, const float (&v)[4]) {
  __stcs(reinterpret_cast<float4*>(dst), make_float4(v[0], v[1], v[2], v[3]));
}

template <typename WT, typename IT, bool PSW, int VB, int MAXV, int UNROLL>
__global__ void __launch_bounds__(256) fwd_gather_kernel(FwdArgs a) {
  using IO = VecIO<WT, VB>;
  using Raw = typename IO::Raw;
  using Acc = typename IO::Acc;
  constexpr int NE = IO::N;  // weight elements per vector
  const unsigned FULL = 0xffffffffu;
  const int lane = lane_id();
  const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;

  for (int64_t u = a.unit_begin + warp0; u < a.unit_end; u += nwarps) {
    const int t = static_cast<int>(u / a.B);
    const int64_t b = u - static_cast<int64_t>(t) * a.B;
    const int col0 = __ldg(a.doff + t);
    const int D = __ldg(a.doff + t + 1) - col0;
    const int64_t E = __ldg(a.roff + t + 1) - __ldg(a.roff + t);
    const Raw* table = reinterpret_cast<const Raw*>(static_cast<const WT*>(a.weights) + __ldg(a.woff + t));
    const int nvec = D / NE;
    const int lpr = nvec >= kWarp ? kWarp : next_pow2_int(nvec);  // lanes per row
    const int rps = kWarp / lpr;                                    // rows per load step
    const int slot = lane / lpr;
    const int vi = lane & (lpr - 1);

    const int64_t s = clamp64(ld_int<IT>(a.offsets, u), 0, a.num_indices);
    const int64_t e = clamp64(ld_int<IT>(a.offsets, u + 1), s, a.num_indices);

    Acc acc[MAXV][NE];
#pragma unroll
    for (int k = 0; k < MAXV; ++k)
#pragma unroll
      for (int i = 0; i < NE; ++i) acc[k][i] = Acc(0);

    for (int64_t base = s; base < e; base += kWarp) {
      const int n = static_cast<int>(min(static_cast<int64_t>(kWarp), e - base));
      int64_t my_id = 0;
      bool my_ok = false;
      float my_w = 1.0f;
      if (lane < n) {
        my_id = ld_int<IT>(a.indices, base + lane);
        my_ok = my_id >= 0 && my_id < E;
        if (PSW) my_w = __ldg(a.psw + base + lane);
        if (!my_ok && a.fused_bounds) {
          static_cast<IT*>(a.indices)[base + lane] = IT(0);
          my_id = 0;
          my_ok = true;
          stat_add(a.stats, TBE_STAT_BAD_INDICES, 1);
        } else if (!my_ok) {
          stat_add(a.stats, TBE_STAT_UNREPAIRED, 1);
        }
      }
      const int32_t row_id = my_ok ? static_cast<int32_t>(my_id) : -1;  // E < 2^31
      for (int j = 0; j < n; j += rps * UNROLL) {
        Raw v[UNROLL][MAXV];
        float w[UNROLL];
#pragma unroll
        for (int q = 0; q < UNROLL; ++q) {
          const int r = j + q * rps + slot;
          const int src = r & (kWarp - 1);
          const int32_t id = __shfl_sync(FULL, row_id, src);
          const bool ok = id >= 0 && r < n;
          w[q] = PSW ? __shfl_sync(FULL, my_w, src) : 1.0f;
          const Raw* row = table + static_cast<int64_t>(ok ? id : 0) * nvec;
#pragma unroll
          for (int k = 0; k < MAXV; ++k) {
            const int vv = vi + k * kWarp;
            if (ok && vv < nvec) v[q][k] = ldg_raw(row + vv);
            else v[q][k] = Raw{};
          }
        }
#pragma unroll
        for (int q = 0; q < UNROLL; ++q) {
#pragma unroll
          for (int k = 0; k < MAXV; ++k) {
            float f[NE];
            IO::unpack(v[q][k], f);
#pragma unroll
            for (int i = 0; i < NE; ++i) {
              if (PSW) acc[k][i] += static_cast<Acc>(f[i]) * static_cast<Acc>(w[q]);
              else acc[k][i] += static_cast<Acc>(f[i]);
            }
          }
        }
      }
    }
    // reduce the row groups of the warp (lanes that share vi)
    for (int m = lpr; m < kWarp; m <<= 1) {
#pragma unroll
      for (int k = 0; k < MAXV; ++k)
#pragma unroll
        for (int i = 0; i < NE; ++i) acc[k][i] += __shfl_xor_sync(FULL, acc[k][i], m);
    }
    if (slot == 0) {
      float* orow = a.out + b * a.total_D + col0;
#pragma unroll
      for (int k = 0; k < MAXV; ++k) {
        const int vv = vi + k * kWarp;
        if (vv < nvec) {
          float o[NE];
#pragma unroll
          for (int i = 0; i < NE; ++i) o[i] = static_cast<float>(acc[k][i]);
          store_out(orow + vv * NE, o);
        }
      }
    }
  }
}

template <typename WT, typename IT, bool PSW, int VB, int MAXV>
cudaError_t launch_t(const FwdArgs& a, const DeviceInfo& dev, cudaStream_t s) {
  constexpr int UNROLL = 4;
  auto k = fwd_gather_kernel<WT, IT, PSW, VB, MAXV, UNROLL>;
  const int threads = 256;
  const int64_t units = a.unit_end - a.unit_begin;
  const int64_t want = (units + (threads / kWarp) - 1) / (threads / kWarp);
  const int grid = persistent_grid(k, threads, 0, dev, want);
  k<<<grid, threads, 0, s>>>(a);
  note_launch();
  return cudaGetLastError();
}

template <typename WT, typename IT, bool PSW, int VB>
cudaError_t dispatch_maxv(const FwdArgs& a, int maxv, const DeviceInfo& dev, cudaStream_t s) {
  switch (maxv) {
    case 1: return launch_t<WT, IT, PSW, VB, 1>(a, dev, s);
    case 2: return launch_t<WT, IT, PSW, VB, 2>(a, dev, s);
    case 4: return launch_t<WT, IT, PSW, VB, 4>(a, dev, s);
    default: return launch_t<WT, IT, PSW, VB, 8>(a, dev, s);
  }
}

template <typename WT, typename IT, bool PSW>
cudaError_t dispatch_vb(const FwdArgs& a, int vb, int maxv, const DeviceInfo& dev, cudaStream_t s) {
  if constexpr (sizeof(WT) == 4) {
    return dispatch_maxv<WT, IT, PSW, 16>(a, maxv, dev, s);
  } else {
    if (vb == 16) return dispatch_maxv<WT, IT, PSW, 16>(a, maxv, dev, s);
    return dispatch_maxv<WT, IT, PSW, 8>(a, maxv, dev, s);
  }
}

template <typename WT>
cudaError_t dispatch_it(const FwdArgs& a, int itype, bool psw, int vb, int maxv,
                        const DeviceInfo& dev, cudaStream_t s) {
  if (itype == TBE_I32) {
    return psw ? dispatch_vb<WT, int32_t, true>(a, vb, maxv, dev, s)
               : dispatch_vb<WT, int32_t, false>(a, vb, maxv, dev, s);
  }
  return psw ? dispatch_vb<WT, int64_t, true>(a, vb, maxv, dev, s)
             : dispatch_vb<WT, int64_t, false>(a, vb, maxv, dev, s);
}

}  // namespace

cudaError_t launch_forward_gather(const Problem& P, const tbe_tables& tab, const void* weights,
                                  void* indices, const void* offsets, const float* psw, float* out,
                                  int64_t unit_begin, int64_t unit_end, bool fused_bounds,
                                  unsigned long long* stats, const DeviceInfo& dev, cudaStream_t s) {
  if (unit_end <= unit_begin) return cudaSuccess;
  FwdArgs a;
  a.weights = weights;
  a.woff = tab.weight_offsets;
  a.doff = tab.D_offsets;
  a.roff = tab.row_offsets;
  a.indices = indices;
  a.offsets = offsets;
  a.psw = psw;
  a.out = out;
  a.B = P.B;
  a.num_indices = P.num_indices;
  a.unit_begin = unit_begin;
  a.unit_end = unit_end;
  a.total_D = P.total_D;
  a.fused_bounds = fused_bounds ? 1 : 0;
  a.stats = stats;
  const int vb = P.vec_bytes;
  const int ne = vb / P.wbytes;
  const int max_nvec = P.max_D / ne;
  int maxv = (max_nvec + kWarp - 1) / kWarp;
  maxv = maxv <= 1 ? 1 : (maxv <= 2 ? 2 : (maxv <= 4 ? 4 : 8));
  const bool has_psw = psw != nullptr;
  switch (P.wdtype) {
    case TBE_F32: return dispatch_it<float>(a, P.itype, has_psw, vb, maxv, dev, s);
    case TBE_F16: return dispatch_it<__half>(a, P.itype, has_psw, vb, maxv, dev, s);
    default: return dispatch_it<__nv_bfloat16>(a, P.itype, has_psw, vb, maxv, dev, s);
  }
}

}  // namespace tbe
