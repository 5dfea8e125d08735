// k_long.cu -- the long-run update (segment length at or above the threshold).
//
// "Modernizing Table Batched Embeddings with FBTriton", section 3: a long run (SL >= 256) is
// split into 256-lookup chunks whose partial sums meet in a workspace, after which either a
// second kernel applies the optimizer or, in one launch, the chunk that sees a countdown reach
// one applies it after a device-scope fence (section 4, Problem 5).
//
// GB300 design: one warp per chunk (rows of the chunk spread over the warp like the forward);
// the chunk sum is merged with float4 atomicAdd (red.global.add.v4.f32) into the run's
// workspace row; fused mode then fences, counts down, and the last warp reads the complete sum
// from L2 and applies the optimizer.
#include "k_update_common.cuh"

namespace tbe {
namespace {

// ------------------------------------------------------------------------------------------
// long runs: chunk partial sums, fused or separate apply
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ int next_pow2_int(int v) { return v <= 1 ? 1 : 1 << (32 - __clz(v - 1)); }

template <typename Acc>
__device__ __forceinline__ void merge_partial(void* ws_row, int vec, const Acc (&a)[4]);
template <>
__device__ __forceinline__ void merge_partial<float>(void* ws_row, int vec, const float (&a)[4]) {
  atomicAdd(reinterpret_cast<float4*>(ws_row) + vec, make_float4(a[0], a[1], a[2], a[3]));
}
template <>
__device__ __forceinline__ void merge_partial<double>(void* ws_row, int vec, const double (&a)[4]) {
  double* p = reinterpret_cast<double*>(ws_row) + 4 * vec;
  atomicAdd(p + 0, a[0]);
  atomicAdd(p + 1, a[1]);
  atomicAdd(p + 2, a[2]);
  atomicAdd(p + 3, a[3]);
}

// Reads a complete workspace row from L2 (bypassing L1) and applies the optimizer with the
// whole warp: lane l owns float4 slices l, l + 32, ...
template <typename WT, int OPT, typename Acc, int MAXV>
__device__ __forceinline__ void apply_from_workspace(const BwdCtx& c, uint32_t key, const void* ws_row) {
  const int t = table_of_row(c.roff, c.T, key);
  const int D = __ldg(c.doff + t + 1) - __ldg(c.doff + t);
  const int nv = D / 4;
  const int lane = lane_id();
  Acc g[MAXV][4];
#pragma unroll
  for (int j = 0; j < MAXV; ++j) {
    const int vec = lane + j * kWarp;
#pragma unroll
    for (int i = 0; i < 4; ++i) g[j][i] = Acc(0);
    if (vec < nv) {
      if constexpr (sizeof(Acc) == 8) {
        const double* p = reinterpret_cast<const double*>(ws_row) + 4 * vec;
#pragma unroll
        for (int i = 0; i < 4; ++i) g[j][i] = __ldcg(p + i);
      } else {
        const float4 f = __ldcg(reinterpret_cast<const float4*>(ws_row) + vec);
        g[j][0] = f.x;
        g[j][1] = f.y;
        g[j][2] = f.z;
        g[j][3] = f.w;
      }
    }
  }
  const int64_t row = static_cast<int64_t>(key) - __ldg(c.roff + t);
  WT* wrow = static_cast<WT*>(c.weights) + __ldg(c.woff + t) + row * D;
  apply_row_group<WT, OPT, Acc, MAXV>(wrow, c.state + key, g, lane, kWarp, nv, D, c.lr, c.eps, FULL);
}

// Sum of one chunk of a long run merged into the run's workspace row; with FUSED, the chunk
// that takes the run's countdown to zero applies the optimizer.
template <typename WT, int FAC, int OPT, int MAXV, bool FUSED>
__device__ __forceinline__ void long_chunk_body(const BwdCtx& c, int64_t ci, const uint32_t* __restrict__ sorted_vals,
                                                const float* __restrict__ sorted_psw, bool merge_bulk,
                                                void* srow) {
  using Acc = typename WTraits<WT>::Acc;
  constexpr bool PSW = FAC != FAC_NONE;  // gradient rows are scaled by a per-lookup factor
  constexpr int UNROLL = 8 / MAXV > 0 ? 8 / MAXV : 1;  // rows in flight per lane: 8 float4 loads
  const int lane = lane_id();
  const size_t row_bytes = static_cast<size_t>(c.max_D) * sizeof(Acc);
    const uint4 rec = __ldg(c.chunks + ci);  // {first lookup, end, key, slot}
    const uint32_t s = rec.x, e = rec.y, key = rec.z, slot = rec.w;
    if (!TBE_GUARD(slot < c.long_cap, c.stats)) return;
    if (!TBE_CHECK(s <= e && e <= c.counters[TBE_CNT_N] && key < c.total_rows, c.stats)) return;
    const int t = table_of_row(c.roff, c.T, key);
    const int col0 = __ldg(c.doff + t);
    const int D = __ldg(c.doff + t + 1) - col0;
    const int nv = D / 4;
    const int lpr = nv >= kWarp ? kWarp : next_pow2_int(nv);
    const int rps = kWarp / lpr;
    const int rs = lane / lpr, vi = lane & (lpr - 1);

    Acc acc[MAXV][4];
#pragma unroll
    for (int j = 0; j < MAXV; ++j)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[j][i] = Acc(0);
    // This lane's float4 slices of the table's columns in bag 0's gradient row.  Lanes whose
    // slice lies past the row width re-read the last slice: their sums are never stored.
    const float4* gbase = reinterpret_cast<const float4*>(c.grad_out + col0);
    const int64_t gstride = c.total_D / 4;  // float4s per gradient row
    int vk[MAXV];
#pragma unroll
    for (int k = 0; k < MAXV; ++k) vk[k] = min(vi + k * kWarp, nv - 1);
    const bool fast = rps * UNROLL <= kWarp;  // a batch never wraps past 32 rows
    const uint32_t last_bag = static_cast<uint32_t>(c.B - 1);
    // The bags of the chunk's lookups, 32 at a time, with the next 32 in flight.  Bags come
    // from the expand step and are < B; the clamp only keeps garbage (offsets that were not
    // repaired) from reading outside grad_out.
    const float* bag_inv = FAC == FAC_INV_LEN ? c.inv_len + static_cast<int64_t>(t) * c.B : nullptr;
    uint32_t nxt_b = 0;
    float nxt_w = 1.f;
    if (s + lane < e) {
      nxt_b = min(__ldg(sorted_vals + s + lane), last_bag);
      if (FAC == FAC_PSW) nxt_w = __ldg(sorted_psw + s + lane);
      if (FAC == FAC_INV_LEN) nxt_w = __ldg(bag_inv + nxt_b);
    }
    for (uint32_t base = s; base < e; base += kWarp) {
      const int n = static_cast<int>(min(static_cast<uint32_t>(kWarp), e - base));
      const uint32_t bag = nxt_b;
      const float my_w = nxt_w;
      nxt_b = 0;
      if (base + kWarp + lane < e) {
        nxt_b = min(__ldg(sorted_vals + base + kWarp + lane), last_bag);
        if (FAC == FAC_PSW) nxt_w = __ldg(sorted_psw + base + kWarp + lane);
        if (FAC == FAC_INV_LEN) nxt_w = __ldg(bag_inv + nxt_b);
      }
      if (fast && n == kWarp) {
        // all 32 rows valid: unpredicated loads
        for (int j = 0; j < kWarp; j += rps * UNROLL) {
          float4 v[UNROLL][MAXV];
          float w[UNROLL];
#pragma unroll
          for (int q = 0; q < UNROLL; ++q) {
            const int rr = j + q * rps + rs;
            const uint32_t b = __shfl_sync(FULL, bag, rr);
            w[q] = PSW ? __shfl_sync(FULL, my_w, rr) : 1.f;
            const float4* grow = gbase + static_cast<int64_t>(b) * gstride;
#pragma unroll
            for (int k = 0; k < MAXV; ++k) v[q][k] = __ldg(grow + vk[k]);
          }
#pragma unroll
          for (int q = 0; q < UNROLL; ++q)
#pragma unroll
            for (int k = 0; k < MAXV; ++k) {
              const Acc wq = static_cast<Acc>(w[q]);
              acc[k][0] += PSW ? static_cast<Acc>(v[q][k].x) * wq : static_cast<Acc>(v[q][k].x);
              acc[k][1] += PSW ? static_cast<Acc>(v[q][k].y) * wq : static_cast<Acc>(v[q][k].y);
              acc[k][2] += PSW ? static_cast<Acc>(v[q][k].z) * wq : static_cast<Acc>(v[q][k].z);
              acc[k][3] += PSW ? static_cast<Acc>(v[q][k].w) * wq : static_cast<Acc>(v[q][k].w);
            }
        }
        continue;
      }
      for (int j = 0; j < n; j += rps * UNROLL) {
        float4 v[UNROLL][MAXV];
        float w[UNROLL];
#pragma unroll
        for (int q = 0; q < UNROLL; ++q) {
          const int rr = j + q * rps + rs;
          const uint32_t b = __shfl_sync(FULL, bag, rr & (kWarp - 1));
          const bool ok = rr < n;
          w[q] = PSW ? __shfl_sync(FULL, my_w, rr & (kWarp - 1)) : 1.f;
          const float4* grow = gbase + static_cast<int64_t>(b) * gstride;
#pragma unroll
          for (int k = 0; k < MAXV; ++k) v[q][k] = ok ? __ldg(grow + vk[k]) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int q = 0; q < UNROLL; ++q)
#pragma unroll
          for (int k = 0; k < MAXV; ++k) {
            const Acc wq = static_cast<Acc>(w[q]);
            acc[k][0] += PSW ? static_cast<Acc>(v[q][k].x) * wq : static_cast<Acc>(v[q][k].x);
            acc[k][1] += PSW ? static_cast<Acc>(v[q][k].y) * wq : static_cast<Acc>(v[q][k].y);
            acc[k][2] += PSW ? static_cast<Acc>(v[q][k].z) * wq : static_cast<Acc>(v[q][k].z);
            acc[k][3] += PSW ? static_cast<Acc>(v[q][k].w) * wq : static_cast<Acc>(v[q][k].w);
          }
      }
    }
    for (int m = lpr; m < kWarp; m <<= 1)
#pragma unroll
      for (int k = 0; k < MAXV; ++k)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[k][i] += __shfl_xor_sync(FULL, acc[k][i], m);
    void* ws_row = static_cast<char*>(c.ws_rows) + static_cast<size_t>(slot) * row_bytes;
    if (merge_bulk) {
      // the chunk sum into this warp's shared-memory row, then one bulk reduction (an
      // asynchronous add of the whole row into the workspace, performed in L2) by lane 0
      if (rs == 0) {
#pragma unroll
        for (int k = 0; k < MAXV; ++k) {
          const int vec = vi + k * kWarp;
          if (vec < nv) {
            if constexpr (sizeof(Acc) == 8) {
              reinterpret_cast<double2*>(srow)[2 * vec] = make_double2(acc[k][0], acc[k][1]);
              reinterpret_cast<double2*>(srow)[2 * vec + 1] = make_double2(acc[k][2], acc[k][3]);
            } else {
              reinterpret_cast<float4*>(srow)[vec] = make_float4(acc[k][0], acc[k][1], acc[k][2], acc[k][3]);
            }
          }
        }
      }
      fence_proxy_async_smem();  // the bulk copy reads the row through the async proxy
      __syncwarp();
      if (lane == 0) bulk_reduce_add<Acc>(ws_row, srow, static_cast<uint32_t>(D * sizeof(Acc)));
      __syncwarp();
    } else if (rs == 0) {
#pragma unroll
      for (int k = 0; k < MAXV; ++k) {
        const int vec = vi + k * kWarp;
        if (vec < nv) merge_partial<Acc>(ws_row, vec, acc[k]);
      }
    }
    if (FUSED) {
      // every lane's partial is visible device-wide before the countdown moves
      __threadfence();
      __syncwarp();
      uint32_t old = 0;
      if (lane == 0) old = atomicSub(c.countdown + slot, 1u);
      old = __shfl_sync(FULL, old, 0);
      if (old == 1) {
        __threadfence();  // acquire: the other chunks' partials, published before their decrements
        apply_from_workspace<WT, OPT, Acc, MAXV>(c, key, ws_row);
      }
    }
}

// Work distribution (tbe_scheduler): GRID = the warps of one resident wave take a fixed stride
// of the chunk list; PERSISTENT = resident warps claim chunks from an atomic counter; CLC = one
// CTA per 8 chunks, whose CTAs, when done, cancel a CTA that has not started yet (cluster launch
// control) and take its chunks instead, so an SM keeps its CTA rather than launching a new one
// ([FBT] section 4, Problem 1, Solution 1.2).
template <typename WT, int FAC, int OPT, int MAXV, bool FUSED>
__global__ void __launch_bounds__(kThreads, 4) long_chunk_kernel(BwdCtx c,
                                                                const uint32_t* __restrict__ sorted_vals,
                                                                const float* __restrict__ sorted_psw,
                                                                int sched, int merge) {
  extern __shared__ __align__(16) uint8_t long_smem[];  // bulk merge: one workspace row per warp
  __shared__ __align__(16) uint4 clc_resp;
  __shared__ __align__(8) uint64_t clc_bar;
  __shared__ int64_t clc_vb;
  using Acc = typename WTraits<WT>::Acc;
  const int lane = lane_id();
  const int wib = threadIdx.x / kWarp, wpb = blockDim.x / kWarp;
  const uint32_t nchunks = min(c.counters[TBE_CNT_CHUNKS], c.chunk_cap);
  const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) / kWarp;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) / kWarp;
  const bool merge_bulk = merge == TBE_MERGE_BULK;
  void* srow = long_smem + static_cast<size_t>(wib) * c.max_D * sizeof(Acc);
  if (sched == TBE_SCHED_CLC) {
    if (threadIdx.x == 0) clc_init(&clc_bar);
    __syncthreads();
  }
  int64_t vb = blockIdx.x;
  uint32_t clc_phase = 0;
  for (int64_t it = 0;; ++it) {
    int64_t ci;
    if (sched == TBE_SCHED_PERSISTENT) {
      uint32_t x = 0;
      if (lane == 0) x = atomicAdd(c.counters + kWorkLong, 1u);
      ci = __shfl_sync(FULL, x, 0);
      if (ci >= nchunks) break;
    } else if (sched == TBE_SCHED_CLC) {
      if (it > 0) {
        if ((vb + 1) * wpb >= nchunks) break;  // later CTAs hold no chunks either (CTA-uniform)
        vb = clc_steal(&clc_resp, &clc_bar, &clc_vb, clc_phase, c.stats);
        if (vb < 0) break;
      }
      ci = vb * wpb + wib;
    } else {
      ci = gw + it * nw;
      if (ci >= nchunks) break;
    }
    if (ci < nchunks) long_chunk_body<WT, FAC, OPT, MAXV, FUSED>(c, ci, sorted_vals, sorted_psw, merge_bulk, srow);
  }
}

template <typename WT, int OPT, int MAXV>
__global__ void __launch_bounds__(kThreads) long_apply_kernel(BwdCtx c) {
  using Acc = typename WTraits<WT>::Acc;
  const uint32_t nlong = min(c.counters[TBE_CNT_LONG], c.long_cap);
  const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) / kWarp;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) / kWarp;
  const size_t row_bytes = static_cast<size_t>(c.max_D) * sizeof(Acc);
  for (int64_t slot = gw; slot < nlong; slot += nw) {
    const uint32_t r = c.long_list[slot];
    const uint32_t key = c.unique[r];
    const void* ws_row = static_cast<const char*>(c.ws_rows) + static_cast<size_t>(slot) * row_bytes;
    apply_from_workspace<WT, OPT, Acc, MAXV>(c, key, ws_row);
  }
}

template <typename WT, int FAC, int OPT, int MAXV>
cudaError_t launch_long_t(const BwdCtx& c, const uint32_t* vals, const float* psw, bool fused, int sched,
                          int merge, const DeviceInfo& dev, cudaStream_t s) {
  using Acc = typename WTraits<WT>::Acc;
  const int64_t want = (static_cast<int64_t>(c.chunk_cap) + (kThreads / kWarp) - 1) / (kThreads / kWarp);
  // bulk merge: one workspace row per warp in shared memory (up to the default 48 KB)
  size_t smem = static_cast<size_t>(kThreads / kWarp) * c.max_D * sizeof(Acc);
  if (merge == TBE_MERGE_BULK && smem > 48 * 1024) merge = TBE_MERGE_ATOMIC;
  if (merge != TBE_MERGE_BULK) smem = 0;
  auto k = fused ? long_chunk_kernel<WT, FAC, OPT, MAXV, true> : long_chunk_kernel<WT, FAC, OPT, MAXV, false>;
  const int64_t resident = persistent_grid(k, kThreads, smem, dev, INT64_MAX);
  int64_t grid;
  if (sched == TBE_SCHED_PERSISTENT) grid = resident;                      // claims from a counter
  else if (sched == TBE_SCHED_CLC) grid = want;                            // one CTA per 8 chunks, stolen when idle
  else grid = resident;                                                    // one resident wave, grid stride
  if (grid > want) grid = want;
  if (grid > 0x7fffffff) grid = 0x7fffffff;
  k<<<static_cast<int>(grid < 1 ? 1 : grid), kThreads, smem, s>>>(c, vals, psw, sched, merge);
  note_launch();
  return cudaGetLastError();
}

template <typename WT, int FAC, int OPT>
cudaError_t launch_long_maxv(const BwdCtx& c, const uint32_t* vals, const float* psw, bool fused, int sched,
                             int merge, int maxv, const DeviceInfo& dev, cudaStream_t s) {
  switch (maxv) {
    case 1: return launch_long_t<WT, FAC, OPT, 1>(c, vals, psw, fused, sched, merge, dev, s);
    case 2: return launch_long_t<WT, FAC, OPT, 2>(c, vals, psw, fused, sched, merge, dev, s);
    case 4: return launch_long_t<WT, FAC, OPT, 4>(c, vals, psw, fused, sched, merge, dev, s);
    default: return launch_long_t<WT, FAC, OPT, 8>(c, vals, psw, fused, sched, merge, dev, s);
  }
}

template <typename WT, int OPT>
cudaError_t launch_apply_maxv(const BwdCtx& c, int maxv, const DeviceInfo& dev, cudaStream_t s) {
  const int64_t want = (static_cast<int64_t>(c.long_cap) + (kThreads / kWarp) - 1) / (kThreads / kWarp);
#define TBE_APPLY_LAUNCH(M)                                          \
  {                                                                  \
    auto k = long_apply_kernel<WT, OPT, M>;                          \
    const int grid = persistent_grid(k, kThreads, 0, dev, want);     \
    k<<<grid, kThreads, 0, s>>>(c);                                  \
    note_launch();                                                   \
    return cudaGetLastError();                                       \
  }
  switch (maxv) {
    case 1: TBE_APPLY_LAUNCH(1)
    case 2: TBE_APPLY_LAUNCH(2)
    case 4: TBE_APPLY_LAUNCH(4)
    default: TBE_APPLY_LAUNCH(8)
  }
#undef TBE_APPLY_LAUNCH
}

}  // namespace

cudaError_t launch_long_updates(const Problem& P, const BwdCtx& c, const BwdLayout& L,
                                tbe_optimizer opt, bool fused, int scheduler, int merge,
                                const DeviceInfo& dev, cudaStream_t s) {
  if (c.long_cap == 0) return cudaSuccess;
  const uint32_t* vals = c.vals[L.final_buf];
  const float* psw = P.scaled ? c.pswbuf[L.final_buf] : nullptr;
  const int maxv = maxv_for(P.max_D);
  return by_weight_type(P.wdtype, [&](auto w) -> cudaError_t {
    using WT = decltype(w);
    if (P.scaled) {
      return opt == TBE_OPT_SGD
                 ? launch_long_maxv<WT, FAC_PSW, TBE_OPT_SGD>(c, vals, psw, fused, scheduler, merge, maxv, dev, s)
                 : launch_long_maxv<WT, FAC_PSW, TBE_OPT_ROWWISE_ADAGRAD>(c, vals, psw, fused, scheduler, merge,
                                                                          maxv, dev, s);
    }
    if (P.mean_inv) {
      return opt == TBE_OPT_SGD
                 ? launch_long_maxv<WT, FAC_INV_LEN, TBE_OPT_SGD>(c, vals, psw, fused, scheduler, merge, maxv, dev, s)
                 : launch_long_maxv<WT, FAC_INV_LEN, TBE_OPT_ROWWISE_ADAGRAD>(c, vals, psw, fused, scheduler, merge,
                                                                              maxv, dev, s);
    }
    return opt == TBE_OPT_SGD
               ? launch_long_maxv<WT, FAC_NONE, TBE_OPT_SGD>(c, vals, psw, fused, scheduler, merge, maxv, dev, s)
               : launch_long_maxv<WT, FAC_NONE, TBE_OPT_ROWWISE_ADAGRAD>(c, vals, psw, fused, scheduler, merge,
                                                                         maxv, dev, s);
  });
}

cudaError_t launch_long_apply(const Problem& P, const BwdCtx& c, const BwdLayout& L,
                              tbe_optimizer opt, const DeviceInfo& dev, cudaStream_t s) {
  (void)L;
  if (c.long_cap == 0) return cudaSuccess;
  const int maxv = maxv_for(P.max_D);
  return by_weight_type(P.wdtype, [&](auto w) -> cudaError_t {
    using WT = decltype(w);
    return opt == TBE_OPT_SGD ? launch_apply_maxv<WT, TBE_OPT_SGD>(c, maxv, dev, s)
                              : launch_apply_maxv<WT, TBE_OPT_ROWWISE_ADAGRAD>(c, maxv, dev, s);
  });
}
}  // namespace tbe
