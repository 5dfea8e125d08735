// k_update.cu -- run classification and the per-row optimizer update.
//
// "Modernizing Table Batched Embeddings with FBTriton":
//   section 3: runs are routed by segment length (SL): a short run (SL < 256) is owned start to
//     finish by one program (gather, accumulate in registers, optimizer, plain store, no
//     atomics); a long run (SL >= 256) is split into 256-lookup chunks whose partial sums meet
//     in a workspace, after which either a second kernel applies the optimizer or, in one
//     launch, the chunk that sees a countdown reach one applies it after a device-scope fence;
//     weighted tables scale each gradient row by its per-sample weight before accumulating.
//   section 4, Problems 3 and 4: short runs are bucketed by next_pow2(D) so each bucket launches
//     with its own width; the classification runs on the device with one atomic per block per
//     list (block counts, one atomicAdd, intra-block offsets), and the consumers read the counts
//     from device memory, so the host never synchronizes.
//   The row-wise Adagrad rule follows "Table-Batched Embeddings in Triton", section 5.
//
// GB300 design:
//   classify   grid-stride over runs; per block, shared-memory counters per list, then one
//              global atomicAdd per non-empty list (and one for chunk descriptors); long runs
//              also get their countdown and a zeroed fp32 workspace row.
//   short run  one group of min(32, D/4) lanes per run (so a warp holds 32/group runs of a
//              narrow bucket); each lane owns float4 slices of the row; the group walks the run's
//              sorted bags, broadcasting them by shuffle, with 4 gradient rows in flight; the
//              optimizer runs in registers and the row is written with plain stores.
//   long run   one warp per chunk (rows of the chunk spread over the warp like the forward);
//              the chunk sum is merged with float4 atomicAdd (red.global.add.v4.f32) into the
//              run's workspace row; fused mode then fences, counts down, and the last warp reads
//              the complete sum from L2 and applies the optimizer.
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
// classify
// ------------------------------------------------------------------------------------------
template <typename Acc>
__global__ void __launch_bounds__(kThreads) classify_kernel(BwdCtx c) {
  __shared__ uint32_t s_cnt[kNumBuckets + 1];
  __shared__ uint32_t s_base[kNumBuckets + 1];
  __shared__ uint32_t s_chunks, s_chunk_base;
  const uint32_t U = min(c.counters[TBE_CNT_RUNS], c.u_cap);
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t r0 = static_cast<int64_t>(blockIdx.x) * blockDim.x; r0 < U; r0 += stride) {
    const int64_t r = r0 + threadIdx.x;
    if (threadIdx.x <= kNumBuckets) s_cnt[threadIdx.x] = 0;
    if (threadIdx.x == 0) s_chunks = 0;
    __syncthreads();
    int list = -1;
    uint32_t nch = 0, my_off = 0, my_choff = 0, len = 0, key = 0, start = 0;
    int D = 0, t = 0;
    if (r < U) {
      key = c.unique[r];
      start = c.run_off[r];
      len = c.run_off[r + 1] - start;
      c.run_len[r] = len;
      if (key < c.total_rows) {
        t = table_of_row(c.roff, c.T, key);
        D = __ldg(c.doff + t + 1) - __ldg(c.doff + t);
        if (len >= static_cast<uint32_t>(c.threshold)) {
          list = kNumBuckets;
          nch = (len + c.chunk - 1) / c.chunk;
          my_choff = atomicAdd(&s_chunks, nch);
        } else {
          list = bucket_of_width(D);
        }
        my_off = atomicAdd(&s_cnt[list], 1u);
      }
    }
    __syncthreads();
    if (threadIdx.x <= kNumBuckets && s_cnt[threadIdx.x] > 0) {
      const int ctr = threadIdx.x == kNumBuckets ? TBE_CNT_LONG : TBE_CNT_SHORT0 + threadIdx.x;
      s_base[threadIdx.x] = atomicAdd(c.counters + ctr, s_cnt[threadIdx.x]);
    }
    if (threadIdx.x == kNumBuckets + 1 && s_chunks > 0)
      s_chunk_base = atomicAdd(c.counters + TBE_CNT_CHUNKS, s_chunks);
    __syncthreads();
    if (list >= 0) {
      const uint32_t slot = s_base[list] + my_off;
      if (list < kNumBuckets) {
        if (slot < c.short_cap[list]) c.short_list[list][slot] = make_uint4(start, len, key, static_cast<uint32_t>(t));
      } else if (slot < c.long_cap) {
        c.long_list[slot] = static_cast<uint32_t>(r);
        c.countdown[slot] = nch;
        float4* row = reinterpret_cast<float4*>(static_cast<Acc*>(c.ws_rows) + static_cast<int64_t>(slot) * c.max_D);
        const int n16 = D * static_cast<int>(sizeof(Acc)) / 16;
        for (int i = 0; i < n16; ++i) row[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        const uint32_t cb = s_chunk_base + my_choff;
        const uint32_t run_end = start + len;
        for (uint32_t k = 0; k < nch; ++k) {
          const uint32_t s0 = start + k * static_cast<uint32_t>(c.chunk);
          const uint32_t e0 = min(s0 + static_cast<uint32_t>(c.chunk), run_end);
          if (cb + k < c.chunk_cap) c.chunks[cb + k] = make_uint4(s0, e0, key, slot);
        }
      }
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------------------------------------
// classify, order-preserving: the lists come out in run (key) order, so consecutive entries --
// and the warps working on them at the same time -- share a table and its slice of grad_out,
// which then stays in L2.  Per-block counts, one scan per list, then each block writes its runs
// at its prefix: one reservation per block per list, intra-block offsets from prefix sums.
// ------------------------------------------------------------------------------------------
constexpr int kLists = kNumBuckets + 2;  // short buckets, long runs, chunks of long runs
constexpr int kLongList = kNumBuckets;
constexpr int kChunkList = kNumBuckets + 1;

__device__ __forceinline__ void cls_segment(uint32_t U, int b, int G, uint32_t* r0, uint32_t* r1) {
  const uint32_t per = ((U + G - 1) / G + kThreads - 1) / kThreads * kThreads;
  *r0 = min(U, static_cast<uint32_t>(b) * per);
  *r1 = min(U, *r0 + per);
}

struct RunRoute {
  int list;  // short bucket, kLongList, or -1 (sentinel run of unrepaired ids)
  uint32_t key, start, len, nch;
  int t, D;
};

__device__ __forceinline__ RunRoute route_run(const BwdCtx& c, uint32_t r) {
  RunRoute x;
  x.key = c.unique[r];
  x.start = c.run_off[r];
  x.len = c.run_off[r + 1] - x.start;
  x.list = -1;
  x.nch = 0;
  x.t = 0;
  x.D = 0;
  if (x.key < c.total_rows) {
    x.t = table_of_row(c.roff, c.T, x.key);
    x.D = __ldg(c.doff + x.t + 1) - __ldg(c.doff + x.t);
    if (x.len >= static_cast<uint32_t>(c.threshold)) {
      x.list = kLongList;
      x.nch = (x.len + c.chunk - 1) / c.chunk;
    } else {
      x.list = bucket_of_width(x.D);
    }
  }
  return x;
}

__global__ void __launch_bounds__(kThreads) classify_count_kernel(BwdCtx c) {
  __shared__ uint32_t s_cnt[kLists];
  if (threadIdx.x < kLists) s_cnt[threadIdx.x] = 0;
  __syncthreads();
  const uint32_t U = min(c.counters[TBE_CNT_RUNS], c.u_cap);
  uint32_t r0, r1;
  cls_segment(U, blockIdx.x, gridDim.x, &r0, &r1);
  for (uint32_t r = r0 + threadIdx.x; r < r1; r += blockDim.x) {
    const RunRoute x = route_run(c, r);
    if (x.list >= 0) atomicAdd(&s_cnt[x.list], 1u);
    if (x.nch) atomicAdd(&s_cnt[kChunkList], x.nch);
  }
  __syncthreads();
  if (threadIdx.x < kLists) c.cls_counts[threadIdx.x * gridDim.x + blockIdx.x] = s_cnt[threadIdx.x];
}

// One CTA per list: exclusive scan of the per-block counts (G <= 1024), total -> counters.
__global__ void __launch_bounds__(1024) list_scan_kernel(BwdCtx c, int G) {
  __shared__ uint32_t s_wsum[32];
  const int lane = lane_id(), w = threadIdx.x / kWarp;
  uint32_t* row = c.cls_counts + blockIdx.x * G;
  const uint32_t v = static_cast<int>(threadIdx.x) < G ? row[threadIdx.x] : 0u;
  uint32_t x = v;
  for (int d = 1; d < kWarp; d <<= 1) {
    const uint32_t o = __shfl_up_sync(FULL, x, d);
    if (lane >= d) x += o;
  }
  if (lane == kWarp - 1) s_wsum[w] = x;
  __syncthreads();
  uint32_t before = 0, total = 0;
  for (int q = 0; q < static_cast<int>(blockDim.x / kWarp); ++q) {
    if (q < w) before += s_wsum[q];
    total += s_wsum[q];
  }
  if (static_cast<int>(threadIdx.x) < G) row[threadIdx.x] = before + x - v;
  if (threadIdx.x == 0) {
    const int l = blockIdx.x;
    const int ctr = l == kChunkList ? TBE_CNT_CHUNKS : (l == kLongList ? TBE_CNT_LONG : TBE_CNT_SHORT0 + l);
    c.counters[ctr] = total;
  }
}

template <typename Acc>
__global__ void __launch_bounds__(kThreads) classify_write_kernel(BwdCtx c) {
  constexpr int W = kThreads / kWarp;
  __shared__ uint32_t s_base[kLists];    // next free entry of each list for this block
  __shared__ uint32_t s_wc[W][kLists];   // per-warp counts (the chunk list holds chunk counts)
  const int lane = lane_id(), w = threadIdx.x / kWarp;
  const unsigned lt = lanemask_lt();
  if (threadIdx.x < kLists) s_base[threadIdx.x] = c.cls_counts[threadIdx.x * gridDim.x + blockIdx.x];
  const uint32_t U = min(c.counters[TBE_CNT_RUNS], c.u_cap);
  uint32_t r0, r1;
  cls_segment(U, blockIdx.x, gridDim.x, &r0, &r1);
  for (uint32_t tb = r0; tb < r1; tb += kThreads) {  // block-uniform
    for (int i = threadIdx.x; i < W * kLists; i += blockDim.x) (&s_wc[0][0])[i] = 0;
    __syncthreads();
    const uint32_t r = tb + threadIdx.x;
    RunRoute x;
    x.list = -1;
    x.nch = 0;
    if (r < r1) {
      x = route_run(c, r);
      c.run_len[r] = x.len;
    }
    // rank among the warp's lanes of the same list; the chunk list by an inclusive scan
    const unsigned peers = __match_any_sync(FULL, static_cast<uint32_t>(x.list));
    const uint32_t rank = __popc(peers & lt);
    if (x.list >= 0 && rank == 0) s_wc[w][x.list] = __popc(peers);
    uint32_t ch = x.nch;
    for (int d = 1; d < kWarp; d <<= 1) {
      const uint32_t o = __shfl_up_sync(FULL, ch, d);
      if (lane >= d) ch += o;
    }
    if (lane == kWarp - 1) s_wc[w][kChunkList] = ch;
    const uint32_t ch_excl = ch - x.nch;
    __syncthreads();
    uint32_t before = 0;  // this warp's prefix in its list within the tile
    if (x.list >= 0)
      for (int q = 0; q < w; ++q) before += s_wc[q][x.list];
    uint32_t ch_before = 0;
    for (int q = 0; q < w; ++q) ch_before += s_wc[q][kChunkList];
    if (x.list >= 0) {
      const uint32_t slot = s_base[x.list] + before + rank;
      if (x.list < kNumBuckets) {
        if (slot < c.short_cap[x.list]) c.short_list[x.list][slot] = make_uint4(x.start, x.len, x.key, static_cast<uint32_t>(x.t));
      } else if (slot < c.long_cap) {
        c.long_list[slot] = r;
        c.countdown[slot] = x.nch;
        float4* row = reinterpret_cast<float4*>(static_cast<Acc*>(c.ws_rows) + static_cast<int64_t>(slot) * c.max_D);
        const int n16 = x.D * static_cast<int>(sizeof(Acc)) / 16;
        for (int i = 0; i < n16; ++i) row[i] = make_float4(0.f, 0.f, 0.f, 0.f);
        const uint32_t cb = s_base[kChunkList] + ch_before + ch_excl;
        const uint32_t run_end = x.start + x.len;
        for (uint32_t k = 0; k < x.nch; ++k) {
          const uint32_t s0 = x.start + k * static_cast<uint32_t>(c.chunk);
          const uint32_t e0 = min(s0 + static_cast<uint32_t>(c.chunk), run_end);
          if (cb + k < c.chunk_cap) c.chunks[cb + k] = make_uint4(s0, e0, x.key, slot);
        }
      }
    }
    __syncthreads();
    if (threadIdx.x < kLists) {  // advance the bases by the tile's totals
      uint32_t tot = 0;
      for (int q = 0; q < W; ++q) tot += s_wc[q][threadIdx.x];
      s_base[threadIdx.x] += tot;
    }
    __syncthreads();
  }
}

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

// ------------------------------------------------------------------------------------------
// short runs
// ------------------------------------------------------------------------------------------
template <typename WT, bool PSW, int OPT, int LPR, int VPL, bool PERSIST>
__global__ void __launch_bounds__(kThreads) short_run_kernel(BwdCtx c, int bucket,
                                                            const uint32_t* __restrict__ sorted_vals,
                                                            const float* __restrict__ sorted_psw) {
  using Acc = typename WTraits<WT>::Acc;
  constexpr int GPW = kWarp / LPR;  // runs per warp
  constexpr int UNROLL = 4;  // gradient rows in flight per run
  const int lane = lane_id();
  const int g = lane / LPR, li = lane % LPR;
  const unsigned gmask = LPR == kWarp ? FULL : (((1u << LPR) - 1u) << (g * LPR));
  const uint32_t count = min(c.counters[TBE_CNT_SHORT0 + bucket], c.short_cap[bucket]);
  const uint4* list = c.short_list[bucket];
  const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) / kWarp;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) / kWarp;
  using IO = VecIO<WT, 4 * sizeof(WT)>;
  using Raw = typename IO::Raw;

  int64_t claim_base = 0, claim_left = 0;
  int64_t it = 0;
  while (true) {
    int64_t base;
    if (PERSIST) {
      if (claim_left == 0) {
        uint32_t b0 = 0;
        if (lane == 0) b0 = atomicAdd(c.counters + kWorkShort0 + bucket, static_cast<uint32_t>(GPW * kClaim));
        claim_base = __shfl_sync(FULL, b0, 0);
        claim_left = kClaim;
      }
      base = claim_base;
      claim_base += GPW;
      --claim_left;
    } else {
      base = (gw + it * nw) * GPW;
      ++it;
    }
    if (base >= count) break;  // warp-uniform
    const int64_t i = base + g;
    uint4 rec = make_uint4(0, 0, 0, 0);  // {first lookup, length, key, table}
    if (i < count) rec = __ldg(list + i);
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
      uint32_t my_b = 0;
      float my_w = 1.f;
      bool my_ok = false;
      if (j0 + li < len) {
        my_b = __ldg(sorted_vals + off + j0 + li);
        if (PSW) my_w = __ldg(sorted_psw + off + j0 + li);
        my_ok = my_b < c.B;
      }
      const int steps = static_cast<int>(min(static_cast<uint32_t>(LPR), maxlen - j0));
      for (int q0 = 0; q0 < steps; q0 += UNROLL) {
        float4 v[UNROLL][VPL];
        float w[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
          const int src = g * LPR + ((q0 + u) & (LPR - 1));
          const uint32_t b = __shfl_sync(FULL, my_b, src);
          const bool ok = __shfl_sync(FULL, static_cast<int>(my_ok), src) && (q0 + u < steps) &&
                          (j0 + q0 + u < len);
          w[u] = PSW ? __shfl_sync(FULL, my_w, src) : 1.f;
          const float4* grow = reinterpret_cast<const float4*>(c.grad_out + static_cast<int64_t>(b) * c.total_D + col0);
#pragma unroll
          for (int jj = 0; jj < VPL; ++jj) {
            const int vec = li + jj * LPR;
            v[u][jj] = (ok && vec < nv) ? __ldg(grow + vec) : make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u)
#pragma unroll
          for (int jj = 0; jj < VPL; ++jj) {
            const Acc wu = static_cast<Acc>(w[u]);
            acc[jj][0] += PSW ? static_cast<Acc>(v[u][jj].x) * wu : static_cast<Acc>(v[u][jj].x);
            acc[jj][1] += PSW ? static_cast<Acc>(v[u][jj].y) * wu : static_cast<Acc>(v[u][jj].y);
            acc[jj][2] += PSW ? static_cast<Acc>(v[u][jj].z) * wu : static_cast<Acc>(v[u][jj].z);
            acc[jj][3] += PSW ? static_cast<Acc>(v[u][jj].w) * wu : static_cast<Acc>(v[u][jj].w);
          }
      }
    }
    if (len > 0) apply_row_prefetched<WT, OPT, Acc, VPL>(wrow, c.state + key, s_old, wv, acc, li, LPR, nv, D,
                                                        c.lr, c.eps, gmask);
  }
}

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

template <typename WT, bool PSW, int OPT, int MAXV, bool FUSED, bool PERSIST>
__global__ void __launch_bounds__(kThreads, 4) long_chunk_kernel(BwdCtx c,
                                                                const uint32_t* __restrict__ sorted_vals,
                                                                const float* __restrict__ sorted_psw) {
  using Acc = typename WTraits<WT>::Acc;
  constexpr int UNROLL = MAXV == 1 ? 8 : 4;  // rows in flight per lane
  const int lane = lane_id();
  const uint32_t nchunks = min(c.counters[TBE_CNT_CHUNKS], c.chunk_cap);
  const int64_t gw = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) / kWarp;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) / kWarp;
  const size_t row_bytes = static_cast<size_t>(c.max_D) * sizeof(Acc);
  int64_t it = 0;
  while (true) {
    int64_t ci;
    if (PERSIST) {
      uint32_t x = 0;
      if (lane == 0) x = atomicAdd(c.counters + kWorkLong, 1u);
      ci = __shfl_sync(FULL, x, 0);
    } else {
      ci = gw + it * nw;
      ++it;
    }
    if (ci >= nchunks) break;
    const uint4 rec = __ldg(c.chunks + ci);  // {first lookup, end, key, slot}
    const uint32_t s = rec.x, e = rec.y, key = rec.z, slot = rec.w;
    if (slot >= c.long_cap) continue;
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
    uint32_t nxt_b = 0;
    float nxt_w = 1.f;
    if (s + lane < e) {
      nxt_b = min(__ldg(sorted_vals + s + lane), last_bag);
      if (PSW) nxt_w = __ldg(sorted_psw + s + lane);
    }
    for (uint32_t base = s; base < e; base += kWarp) {
      const int n = static_cast<int>(min(static_cast<uint32_t>(kWarp), e - base));
      const uint32_t bag = nxt_b;
      const float my_w = nxt_w;
      nxt_b = 0;
      if (base + kWarp + lane < e) {
        nxt_b = min(__ldg(sorted_vals + base + kWarp + lane), last_bag);
        if (PSW) nxt_w = __ldg(sorted_psw + base + kWarp + lane);
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
    if (rs == 0) {
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

// ------------------------------------------------------------------------------------------
// dispatch
// ------------------------------------------------------------------------------------------
template <typename WT, bool PSW, int OPT, int LPR, int VPL>
cudaError_t launch_short_t(const BwdCtx& c, int bucket, const uint32_t* vals, const float* psw,
                           bool persist, const DeviceInfo& dev, cudaStream_t s) {
  constexpr int GPW = kWarp / LPR;
  const int64_t groups_per_cta = (kThreads / kWarp) * GPW;
  const int64_t want = (static_cast<int64_t>(c.short_cap[bucket]) + groups_per_cta - 1) / groups_per_cta;
  if (persist) {
    auto k = short_run_kernel<WT, PSW, OPT, LPR, VPL, true>;
    const int grid = persistent_grid(k, kThreads, 0, dev, want);
    k<<<grid, kThreads, 0, s>>>(c, bucket, vals, psw);
    note_launch();
  } else {
    auto k = short_run_kernel<WT, PSW, OPT, LPR, VPL, false>;
    // sixteen waves of CTAs (capped by the list capacity): CTAs that finish early hand their SM
    // to the next, which evens out runs of uneven length better than one resident wave
    const int64_t g16 = static_cast<int64_t>(persistent_grid(k, kThreads, 0, dev, INT64_MAX)) * 16;
    const int grid = static_cast<int>(g16 < want ? g16 : want);
    k<<<grid, kThreads, 0, s>>>(c, bucket, vals, psw);
    note_launch();
  }
  return cudaGetLastError();
}

template <typename WT, bool PSW, int OPT>
cudaError_t launch_short_bucket(const BwdCtx& c, int bucket, const uint32_t* vals, const float* psw,
                                bool persist, const DeviceInfo& dev, cudaStream_t s) {
  // next_pow2(D) = 2^bucket; float4 slices per row = 2^(bucket-2): min(32, slices) lanes per run
  switch (bucket) {
    case 2: return launch_short_t<WT, PSW, OPT, 1, 1>(c, bucket, vals, psw, persist, dev, s);
    case 3: return launch_short_t<WT, PSW, OPT, 2, 1>(c, bucket, vals, psw, persist, dev, s);
    case 4: return launch_short_t<WT, PSW, OPT, 4, 1>(c, bucket, vals, psw, persist, dev, s);
    case 5: return launch_short_t<WT, PSW, OPT, 8, 1>(c, bucket, vals, psw, persist, dev, s);
    case 6: return launch_short_t<WT, PSW, OPT, 16, 1>(c, bucket, vals, psw, persist, dev, s);
    case 7: return launch_short_t<WT, PSW, OPT, 32, 1>(c, bucket, vals, psw, persist, dev, s);
    case 8: return launch_short_t<WT, PSW, OPT, 32, 2>(c, bucket, vals, psw, persist, dev, s);
    case 9: return launch_short_t<WT, PSW, OPT, 32, 4>(c, bucket, vals, psw, persist, dev, s);
    case 10: return launch_short_t<WT, PSW, OPT, 32, 8>(c, bucket, vals, psw, persist, dev, s);
    default: return cudaErrorInvalidValue;
  }
}

template <typename WT, bool PSW, int OPT, int MAXV>
cudaError_t launch_long_t(const BwdCtx& c, const uint32_t* vals, const float* psw, bool fused,
                          bool persist, const DeviceInfo& dev, cudaStream_t s) {
  const int64_t want = (static_cast<int64_t>(c.chunk_cap) + (kThreads / kWarp) - 1) / (kThreads / kWarp);
#define TBE_LONG_LAUNCH(F, P)                                            \
  {                                                                      \
    auto k = long_chunk_kernel<WT, PSW, OPT, MAXV, F, P>;                \
    const int grid = persistent_grid(k, kThreads, 0, dev, want);         \
    k<<<grid, kThreads, 0, s>>>(c, vals, psw);                           \
    note_launch();                                                   \
  }
  if (fused) {
    if (persist) TBE_LONG_LAUNCH(true, true) else TBE_LONG_LAUNCH(true, false)
  } else {
    if (persist) TBE_LONG_LAUNCH(false, true) else TBE_LONG_LAUNCH(false, false)
  }
#undef TBE_LONG_LAUNCH
  return cudaGetLastError();
}

template <typename WT, bool PSW, int OPT>
cudaError_t launch_long_maxv(const BwdCtx& c, const uint32_t* vals, const float* psw, bool fused,
                             bool persist, int maxv, const DeviceInfo& dev, cudaStream_t s) {
  switch (maxv) {
    case 1: return launch_long_t<WT, PSW, OPT, 1>(c, vals, psw, fused, persist, dev, s);
    case 2: return launch_long_t<WT, PSW, OPT, 2>(c, vals, psw, fused, persist, dev, s);
    case 4: return launch_long_t<WT, PSW, OPT, 4>(c, vals, psw, fused, persist, dev, s);
    default: return launch_long_t<WT, PSW, OPT, 8>(c, vals, psw, fused, persist, dev, s);
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

cudaError_t launch_classify(const Problem& P, const BwdCtx& c, const DeviceInfo& dev, int mode, cudaStream_t s) {
  if (mode == TBE_CLASSIFY_ATOMIC) {  // one atomicAdd per block per list: list order is arbitrary
    const int64_t want = (static_cast<int64_t>(c.u_cap) + kThreads - 1) / kThreads;
    if (P.wdtype == TBE_F32) {  // fp64 workspace rows for fp32 tables
      const int grid = persistent_grid(classify_kernel<double>, kThreads, 0, dev, want);
      classify_kernel<double><<<grid, kThreads, 0, s>>>(c);
    } else {
      const int grid = persistent_grid(classify_kernel<float>, kThreads, 0, dev, want);
      classify_kernel<float><<<grid, kThreads, 0, s>>>(c);
    }
    note_launch();
    return cudaGetLastError();
  }
  const int G = c.cls_grid;
  classify_count_kernel<<<G, kThreads, 0, s>>>(c);
  note_launch();
  list_scan_kernel<<<kLists, 1024, 0, s>>>(c, G);
  note_launch();
  if (P.wdtype == TBE_F32) classify_write_kernel<double><<<G, kThreads, 0, s>>>(c);
  else classify_write_kernel<float><<<G, kThreads, 0, s>>>(c);
  note_launch();
  return cudaGetLastError();
}

cudaError_t launch_short_updates(const Problem& P, const BwdCtx& c, const BwdLayout& L,
                                 tbe_optimizer opt, int scheduler, const DeviceInfo& dev,
                                 cudaStream_t s) {
  const uint32_t* vals = c.vals[L.final_buf];
  const float* psw = P.weighted ? c.pswbuf[L.final_buf] : nullptr;
  const bool persist = scheduler == TBE_SCHED_PERSISTENT;
  for (int k = 2; k < kNumBuckets; ++k) {
    if (c.short_cap[k] == 0) continue;
    cudaError_t e = by_weight_type(P.wdtype, [&](auto w) -> cudaError_t {
      using WT = decltype(w);
      if (P.weighted) {
        return opt == TBE_OPT_SGD ? launch_short_bucket<WT, true, TBE_OPT_SGD>(c, k, vals, psw, persist, dev, s)
                                  : launch_short_bucket<WT, true, TBE_OPT_ROWWISE_ADAGRAD>(c, k, vals, psw, persist, dev, s);
      }
      return opt == TBE_OPT_SGD ? launch_short_bucket<WT, false, TBE_OPT_SGD>(c, k, vals, psw, persist, dev, s)
                                : launch_short_bucket<WT, false, TBE_OPT_ROWWISE_ADAGRAD>(c, k, vals, psw, persist, dev, s);
    });
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_long_updates(const Problem& P, const BwdCtx& c, const BwdLayout& L,
                                tbe_optimizer opt, bool fused, int scheduler, const DeviceInfo& dev,
                                cudaStream_t s) {
  if (c.long_cap == 0) return cudaSuccess;
  const uint32_t* vals = c.vals[L.final_buf];
  const float* psw = P.weighted ? c.pswbuf[L.final_buf] : nullptr;
  const bool persist = scheduler == TBE_SCHED_PERSISTENT;
  const int maxv = maxv_for(P.max_D);
  return by_weight_type(P.wdtype, [&](auto w) -> cudaError_t {
    using WT = decltype(w);
    if (P.weighted) {
      return opt == TBE_OPT_SGD ? launch_long_maxv<WT, true, TBE_OPT_SGD>(c, vals, psw, fused, persist, maxv, dev, s)
                                : launch_long_maxv<WT, true, TBE_OPT_ROWWISE_ADAGRAD>(c, vals, psw, fused, persist, maxv, dev, s);
    }
    return opt == TBE_OPT_SGD ? launch_long_maxv<WT, false, TBE_OPT_SGD>(c, vals, psw, fused, persist, maxv, dev, s)
                              : launch_long_maxv<WT, false, TBE_OPT_ROWWISE_ADAGRAD>(c, vals, psw, fused, persist, maxv, dev, s);
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
