// k_classify.cu -- the on-device run classifier.
//
// "Modernizing Table Batched Embeddings with FBTriton", section 4, Problems 3 and 4: short runs
// are bucketed by next_pow2(D) so each bucket launches with its own width; the classification
// runs on the device with one atomic per block per list (block counts, one atomicAdd,
// intra-block offsets from prefix sums), and the consumers read the counts from device memory,
// so the host never synchronizes.  Section 3: runs of at least the threshold (256) are split
// into 256-lookup chunks whose partial sums meet in a workspace row.
//
// GB300 design: grid-stride over runs; per block, shared-memory counters per list, then one
// global atomicAdd per non-empty list (and one for chunk descriptors); long runs also get their
// countdown and a zeroed workspace row.  The order-preserving option replaces the atomics with
// per-block counts and one scan per list, so the lists come out in key order.
#include "k_update_common.cuh"

namespace tbe {
namespace {

// ------------------------------------------------------------------------------------------
// classify
// ------------------------------------------------------------------------------------------
template <typename Acc>
__global__ void __launch_bounds__(kThreads) classify_kernel(BwdCtx c) {
  __shared__ uint32_t s_cnt[kNumBuckets + 1];
  __shared__ uint32_t s_base[kNumBuckets + 1];
  __shared__ uint32_t s_chunks, s_chunk_base;
  const uint32_t U = min(c.counters[TBE_CNT_RUNS], c.u_cap);
  const uint32_t N = c.counters[TBE_CNT_N];
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
      const uint32_t end = c.run_off[r + 1];
      len = end - start;
      c.run_len[r] = len;
      if (key < c.total_rows && TBE_CHECK(start <= end && end <= N, c.stats)) {
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
        if (TBE_GUARD(slot < c.short_cap[list], c.stats))
          c.short_list[list][slot] = make_uint4(start, len, key, static_cast<uint32_t>(t));
      } else if (TBE_GUARD(slot < c.long_cap, c.stats)) {
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
          if (TBE_GUARD(cb + k < c.chunk_cap, c.stats)) c.chunks[cb + k] = make_uint4(s0, e0, key, slot);
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

// The route of the run with linear key `key` covering sorted positions [start, end) of the N.
__device__ __forceinline__ RunRoute route_of(const BwdCtx& c, uint32_t key, uint32_t start, uint32_t end,
                                             uint32_t N) {
  RunRoute x;
  x.key = key;
  x.start = start;
  x.len = end - start;
  x.list = -1;
  x.nch = 0;
  x.t = 0;
  x.D = 0;
  if (x.key < c.total_rows && TBE_CHECK(start <= end && end <= N, c.stats)) {
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

__device__ __forceinline__ RunRoute route_run(const BwdCtx& c, uint32_t r, uint32_t N) {
  return route_of(c, c.unique[r], c.run_off[r], c.run_off[r + 1], N);
}

__global__ void __launch_bounds__(kThreads) classify_count_kernel(BwdCtx c) {
  __shared__ uint32_t s_cnt[kLists];
  if (threadIdx.x < kLists) s_cnt[threadIdx.x] = 0;
  __syncthreads();
  const uint32_t U = min(c.counters[TBE_CNT_RUNS], c.u_cap);
  const uint32_t N = c.counters[TBE_CNT_N];
  uint32_t r0, r1;
  cls_segment(U, blockIdx.x, gridDim.x, &r0, &r1);
#pragma unroll 4
  for (uint32_t r = r0 + threadIdx.x; r < r1; r += blockDim.x) {
    const RunRoute x = route_run(c, r, N);
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
  const uint32_t N = c.counters[TBE_CNT_N];
  uint32_t r0, r1;
  cls_segment(U, blockIdx.x, gridDim.x, &r0, &r1);
  // this thread's run of the next tile (key, start, end), loaded while the current tile is
  // ranked and written, so a tile's run records are not one DRAM round trip on its own path
  uint32_t nkey = 0, nstart = 0, nend = 0;
  auto fetch = [&](uint32_t r) {
    if (r < r1) {
      nkey = c.unique[r];
      nstart = c.run_off[r];
      nend = c.run_off[r + 1];
    }
  };
  fetch(r0 + threadIdx.x);
  for (uint32_t tb = r0; tb < r1; tb += kThreads) {  // block-uniform
    const uint32_t key = nkey, start = nstart, end = nend;
    fetch(tb + kThreads + threadIdx.x);
    for (int i = threadIdx.x; i < W * kLists; i += blockDim.x) (&s_wc[0][0])[i] = 0;
    __syncthreads();
    const uint32_t r = tb + threadIdx.x;
    RunRoute x;
    x.list = -1;
    x.nch = 0;
    if (r < r1) {
      x = route_of(c, key, start, end, N);
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
        if (TBE_GUARD(slot < c.short_cap[x.list], c.stats))
          c.short_list[x.list][slot] = make_uint4(x.start, x.len, x.key, static_cast<uint32_t>(x.t));
      } else if (TBE_GUARD(slot < c.long_cap, c.stats)) {
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
          if (TBE_GUARD(cb + k < c.chunk_cap, c.stats)) c.chunks[cb + k] = make_uint4(s0, e0, x.key, slot);
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
}  // namespace tbe
