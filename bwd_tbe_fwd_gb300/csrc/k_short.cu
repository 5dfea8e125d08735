// k_short.cu -- the short-run update (segment length below the threshold).
//
// "Modernizing Table Batched Embeddings with FBTriton", section 3: a short run (SL < 256) is
// owned start to finish by one program -- gather, accumulate in registers, optimizer, plain
// store, no atomics; weighted tables scale each gradient row by its per-sample weight before
// accumulating.  Section 4, Problem 3: one launch per next_pow2(D) bucket, each with its own width.
//
// GB300 design: one group of min(32, D/4) lanes per run (a warp holds 32/group runs of a narrow
// bucket); each lane owns float4 slices of the row; the run's weight row and state are fetched
// before its gradient rows (and, for unweighted tables, the next claimed run's record meanwhile);
// the group walks the run's sorted bags, broadcasting them by shuffle, in batches of up to 4
// gradient rows that never run past the run; the optimizer runs in registers and the row is
// written with plain stores.
#include "k_update_common.cuh"

namespace tbe {
namespace {

// ------------------------------------------------------------------------------------------
// short runs
// ------------------------------------------------------------------------------------------
constexpr uint32_t kNoBag = 0xffffffffu;  // B < 2^31: never a bag id

template <typename WT, int FAC, int OPT, int LPR, int VPL, bool PERSIST>
__global__ void __launch_bounds__(kThreads) short_run_kernel(BwdCtx c, int bucket,
                                                            const uint32_t* __restrict__ sorted_vals,
                                                            const float* __restrict__ sorted_psw) {
  using Acc = typename WTraits<WT>::Acc;
  constexpr int GPW = kWarp / LPR;  // runs per warp
  const int lane = lane_id();
  const int g = lane / LPR, li = lane % LPR;
  const unsigned gmask = LPR == kWarp ? FULL : (((1u << LPR) - 1u) << (g * LPR));
  const uint32_t count = min(c.counters[TBE_CNT_SHORT0 + bucket], c.short_cap[bucket]);
  const uint4* list = c.short_list[bucket];
  const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) / kWarp;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) / kWarp;
  using IO = VecIO<WT, 4 * sizeof(WT)>;
  using Raw = typename IO::Raw;
  constexpr bool PSW = FAC != FAC_NONE;  // gradient rows are scaled by a per-lookup factor

  // Unweighted tables fetch the next claimed run's record while the current run is updated
  // (stress batch: short stage 1.13 -> 1.04 ms); with per-lookup factors that measured slower.
  constexpr bool PREFETCH = !PSW;
  int64_t claim_base = 0, claim_left = 0;
  int64_t it = 0;
  auto next_base = [&]() -> int64_t {  // warp-uniform
    int64_t b;
    if (PERSIST) {
      if (claim_left == 0) {
        uint32_t b0 = 0;
        if (lane == 0) b0 = atomicAdd(c.counters + kWorkShort0 + bucket, static_cast<uint32_t>(GPW * kClaim));
        claim_base = __shfl_sync(FULL, b0, 0);
        claim_left = kClaim;
      }
      b = claim_base;
      claim_base += GPW;
      --claim_left;
    } else {
      b = (gw + it * nw) * GPW;
      ++it;
    }
    return b;
  };
  int64_t base = next_base();
  uint4 nrec = make_uint4(0, 0, 0, 0);
  if (PREFETCH && base + g < count) nrec = __ldg(list + base + g);
  while (base < count) {  // warp-uniform
    const int64_t i = base + g;
    uint4 rec = make_uint4(0, 0, 0, 0);  // {first lookup, length, key, table}
    if constexpr (PREFETCH) {
      const uint4 fetched = nrec;
      base = next_base();
      nrec = make_uint4(0, 0, 0, 0);
      if (base + g < count) nrec = __ldg(list + base + g);
      if (i < count) rec = fetched;
    } else {
      if (i < count) rec = __ldg(list + i);
    }
    if (i < count && !TBE_CHECK(rec.w < static_cast<uint32_t>(c.T) && rec.z < c.total_rows &&
                                    rec.x <= c.counters[TBE_CNT_N] && rec.y <= c.counters[TBE_CNT_N] - rec.x,
                                c.stats))
      rec = make_uint4(0, 0, 0, 0);  // skipped: no row read or written
    const uint32_t off = rec.x, len = rec.y, key = rec.z;
    const int t = static_cast<int>(rec.w);
    const int col0 = __ldg(c.doff + t);
    const int D = __ldg(c.doff + t + 1) - col0;
    const int nv = D / 4;
    const uint32_t maxlen = __reduce_max_sync(FULL, len);

    // the row and its state do not depend on the gradient: fetch them first
    WT* wrow = static_cast<WT*>(c.weights) + __ldg(c.woff + t) +
               (static_cast<int64_t>(key) - __ldg(c.roff + t)) * D;
    Raw wv[VPL];
#pragma unroll
    for (int j = 0; j < VPL; ++j) {
      const int vec = li + j * LPR;
      wv[j] = (len > 0 && vec < nv) ? reinterpret_cast<const Raw*>(wrow)[vec] : Raw{};
    }
    float s_old = 0.f;
    if (OPT == TBE_OPT_ROWWISE_ADAGRAD && len > 0) s_old = c.state[key];

    Acc acc[VPL][4];
#pragma unroll
    for (int j = 0; j < VPL; ++j)
#pragma unroll
      for (int q = 0; q < 4; ++q) acc[j][q] = Acc(0);

    for (uint32_t j0 = 0; j0 < maxlen; j0 += LPR) {
      // this lane's lookup of the window: its bag (kNoBag past the run, or for a bag id outside
      // the batch, which only offsets left unrepaired can give: no row is read) and its factor
      uint32_t my_b = kNoBag;
      float my_w = 1.f;
      if (j0 + li < len) {
        my_b = __ldg(sorted_vals + off + j0 + li);
        if (my_b >= static_cast<uint32_t>(c.B)) my_b = kNoBag;
        if (FAC == FAC_PSW) my_w = __ldg(sorted_psw + off + j0 + li);
        if (FAC == FAC_INV_LEN && my_b != kNoBag) my_w = __ldg(c.inv_len + static_cast<int64_t>(t) * c.B + my_b);
      }
      const int steps = static_cast<int>(min(static_cast<uint32_t>(LPR), maxlen - j0));
      auto rows = [&](auto uc, int q0) {
        constexpr int U = decltype(uc)::value;
        float4 v[U][VPL];
        float w[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int src = g * LPR + ((q0 + u) & (LPR - 1));
          const uint32_t b = __shfl_sync(FULL, my_b, src);
          const bool ok = b != kNoBag && q0 + u < steps;
          const float4* grow = reinterpret_cast<const float4*>(c.grad_out + static_cast<int64_t>(b) * c.total_D + col0);
#pragma unroll
          for (int jj = 0; jj < VPL; ++jj) {
            const int vec = li + jj * LPR;
            v[u][jj] = (ok && vec < nv) ? __ldg(grow + vec) : make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
        // the factors after the row loads: with FAC_INV_LEN each one is a load that depends on
        // the bag, which must not hold the row loads back
#pragma unroll
        for (int u = 0; u < U; ++u) w[u] = PSW ? __shfl_sync(FULL, my_w, g * LPR + ((q0 + u) & (LPR - 1))) : 1.f;
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
          for (int jj = 0; jj < VPL; ++jj) {
            const Acc wu = static_cast<Acc>(w[u]);
            acc[jj][0] += PSW ? static_cast<Acc>(v[u][jj].x) * wu : static_cast<Acc>(v[u][jj].x);
            acc[jj][1] += PSW ? static_cast<Acc>(v[u][jj].y) * wu : static_cast<Acc>(v[u][jj].y);
            acc[jj][2] += PSW ? static_cast<Acc>(v[u][jj].z) * wu : static_cast<Acc>(v[u][jj].z);
            acc[jj][3] += PSW ? static_cast<Acc>(v[u][jj].w) * wu : static_cast<Acc>(v[u][jj].w);
          }
      };
      // Rows in flight: most runs are a few lookups long, so a batch must not carry steps past the
      // run.  Unweighted tables take batches of 4 while 4 remain, then 2, then 1; with per-lookup
      // factors batches of 2 (the factor loads' registers) measured faster.
      int q0 = 0;
      if constexpr (PSW) {
        for (; q0 < steps; q0 += 2) rows(std::integral_constant<int, 2>{}, q0);
      } else {
        for (; q0 + 4 <= steps; q0 += 4) rows(std::integral_constant<int, 4>{}, q0);
        for (; q0 + 2 <= steps; q0 += 2) rows(std::integral_constant<int, 2>{}, q0);
        if (q0 < steps) rows(std::integral_constant<int, 1>{}, q0);
      }
    }
    if (len > 0) apply_row_prefetched<WT, OPT, Acc, VPL>(wrow, c.state + key, s_old, wv, acc, li, LPR, nv, D,
                                                        c.lr, c.eps, gmask);
    if constexpr (!PREFETCH) base = next_base();
  }
}

template <typename WT, int FAC, int OPT, int LPR, int VPL>
cudaError_t launch_short_t(const BwdCtx& c, int bucket, const uint32_t* vals, const float* psw,
                           bool persist, const DeviceInfo& dev, cudaStream_t s) {
  constexpr int GPW = kWarp / LPR;
  const int64_t groups_per_cta = (kThreads / kWarp) * GPW;
  const int64_t want = (static_cast<int64_t>(c.short_cap[bucket]) + groups_per_cta - 1) / groups_per_cta;
  if (persist) {
    auto k = short_run_kernel<WT, FAC, OPT, LPR, VPL, true>;
    const int grid = persistent_grid(k, kThreads, 0, dev, want);
    k<<<grid, kThreads, 0, s>>>(c, bucket, vals, psw);
    note_launch();
  } else {
    auto k = short_run_kernel<WT, FAC, OPT, LPR, VPL, false>;
    // sixteen waves of CTAs (capped by the list capacity): CTAs that finish early hand their SM
    // to the next, which evens out runs of uneven length better than one resident wave
    const int64_t g16 = static_cast<int64_t>(persistent_grid(k, kThreads, 0, dev, INT64_MAX)) * 16;
    const int grid = static_cast<int>(g16 < want ? g16 : want);
    k<<<grid, kThreads, 0, s>>>(c, bucket, vals, psw);
    note_launch();
  }
  return cudaGetLastError();
}

template <typename WT, int FAC, int OPT>
cudaError_t launch_short_bucket(const BwdCtx& c, int bucket, const uint32_t* vals, const float* psw,
                                bool persist, const DeviceInfo& dev, cudaStream_t s) {
  // next_pow2(D) = 2^bucket; float4 slices per row = 2^(bucket-2): min(32, slices) lanes per run
  switch (bucket) {
    case 2: return launch_short_t<WT, FAC, OPT, 1, 1>(c, bucket, vals, psw, persist, dev, s);
    case 3: return launch_short_t<WT, FAC, OPT, 2, 1>(c, bucket, vals, psw, persist, dev, s);
    case 4: return launch_short_t<WT, FAC, OPT, 4, 1>(c, bucket, vals, psw, persist, dev, s);
    case 5: return launch_short_t<WT, FAC, OPT, 8, 1>(c, bucket, vals, psw, persist, dev, s);
    case 6: return launch_short_t<WT, FAC, OPT, 16, 1>(c, bucket, vals, psw, persist, dev, s);
    case 7: return launch_short_t<WT, FAC, OPT, 32, 1>(c, bucket, vals, psw, persist, dev, s);
    case 8: return launch_short_t<WT, FAC, OPT, 32, 2>(c, bucket, vals, psw, persist, dev, s);
    case 9: return launch_short_t<WT, FAC, OPT, 32, 4>(c, bucket, vals, psw, persist, dev, s);
    case 10: return launch_short_t<WT, FAC, OPT, 32, 8>(c, bucket, vals, psw, persist, dev, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_short_updates(const Problem& P, const BwdCtx& c, const BwdLayout& L,
                                 tbe_optimizer opt, int scheduler, const DeviceInfo& dev,
                                 cudaStream_t s) {
  const uint32_t* vals = c.vals[L.final_buf];
  const float* psw = P.scaled ? c.pswbuf[L.final_buf] : nullptr;
  const bool persist = scheduler == TBE_SCHED_PERSISTENT;
  for (int k = 2; k < kNumBuckets; ++k) {
    if (c.short_cap[k] == 0) continue;
    cudaError_t e = by_weight_type(P.wdtype, [&](auto w) -> cudaError_t {
      using WT = decltype(w);
      if (P.scaled) {
        return opt == TBE_OPT_SGD ? launch_short_bucket<WT, FAC_PSW, TBE_OPT_SGD>(c, k, vals, psw, persist, dev, s)
                                  : launch_short_bucket<WT, FAC_PSW, TBE_OPT_ROWWISE_ADAGRAD>(c, k, vals, psw, persist, dev, s);
      }
      if (P.mean_inv) {
        return opt == TBE_OPT_SGD ? launch_short_bucket<WT, FAC_INV_LEN, TBE_OPT_SGD>(c, k, vals, psw, persist, dev, s)
                                  : launch_short_bucket<WT, FAC_INV_LEN, TBE_OPT_ROWWISE_ADAGRAD>(c, k, vals, psw, persist, dev, s);
      }
      return opt == TBE_OPT_SGD ? launch_short_bucket<WT, FAC_NONE, TBE_OPT_SGD>(c, k, vals, psw, persist, dev, s)
                                : launch_short_bucket<WT, FAC_NONE, TBE_OPT_ROWWISE_ADAGRAD>(c, k, vals, psw, persist, dev, s);
    });
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}
}  // namespace tbe
