// k_sort.cu -- transpose of the batch into runs: linearize, sort, run-length encode.
//
// "Modernizing Table Batched Embeddings with FBTriton", section 3: transpose_embedding_input
// turns the batch (which rows each sample read) into runs (which samples read each row):
// every lookup's (table, row) becomes one linear key, the keys are sorted, and equal keys form
// one run.  "Table-Batched Embeddings in Triton", section 2, spells the steps out: linear key =
// first row of the table + id, a stable sort, then run-length encoding into unique keys,
// lengths and start offsets.
//
// GB300 design:
//   expand      one CTA per 512 consecutive bags; their lookups are one contiguous range, read
//               coalesced; each lookup finds its bag by binary search over the CTA's offsets in
//               shared memory and writes key = row_offsets[t] + id (uint32) and its bag b
//               (plus its per-sample weight when weighted).
//   radix sort  LSD, 8-bit digits, as many passes as the key range needs (ceil(bits/8), the
//               range being sum E + 1 for an out-of-range sentinel).  Each pass is
//               reduce-then-scan: a per-CTA digit histogram over a contiguous segment, one
//               exclusive scan of the [digit][CTA] counts, and a stable scatter in which each
//               CTA walks its segment in 4096-key tiles, ranks keys with warp-level match
//               (__match_any_sync) and per-warp digit counters in shared memory, reorders the
//               tile in shared memory and writes each digit's keys as one contiguous run.
//               No CTA ever waits on another, so the sort needs no spin loops.
//   RLE         two passes over the sorted keys: per-CTA head counts, then each CTA writes the
//               unique keys and run starts of its segment at its prefix of the counts.
#include <atomic>

#include "tbe_internal.cuh"

namespace tbe {
namespace {

constexpr int kThreads = 256;
constexpr unsigned FULL = 0xffffffffu;

// ------------------------------------------------------------------------------------------
// expand
// ------------------------------------------------------------------------------------------
struct ExpandArgs {
  const void* indices;
  const void* offsets;
  const float* psw;
  const int64_t* roff;
  int64_t B, TB, num_indices;
  uint32_t sentinel;  // key of an out-of-range id: sum of E (sorts after every real row)
  uint32_t* keys;
  uint32_t* vals;
  float* psw_out;
  uint32_t* counters;
  unsigned long long* stats;
};

template <typename IT, bool PSW>
__global__ void __launch_bounds__(kThreads) expand_kernel(ExpandArgs a) {
  __shared__ int64_t s_off[kExpandBags + 1];
  __shared__ unsigned long long s_bad;
  const int64_t N = clamp64(ld_int<IT>(a.offsets, a.TB), 0, a.num_indices);
  const int64_t i0 = static_cast<int64_t>(blockIdx.x) * kExpandBags;
  const int nb = static_cast<int>(min(static_cast<int64_t>(kExpandBags), a.TB - i0));
  if (threadIdx.x == 0) {
    s_bad = 0;
    if (blockIdx.x == 0) a.counters[TBE_CNT_N] = static_cast<uint32_t>(N);
  }
  for (int k = threadIdx.x; k <= nb; k += blockDim.x) s_off[k] = clamp64(ld_int<IT>(a.offsets, i0 + k), 0, N);
  __syncthreads();
  unsigned long long bad = 0;
  if (threadIdx.x < nb && s_off[threadIdx.x + 1] < s_off[threadIdx.x]) ++bad;  // decreasing offsets
  for (int k = threadIdx.x + kThreads; k < nb; k += blockDim.x)
    if (s_off[k + 1] < s_off[k]) ++bad;
  const int64_t t0 = a.B > 0 ? i0 / a.B : 0;
  const int64_t r0 = i0 - t0 * a.B;
  const uint32_t B32 = static_cast<uint32_t>(a.B);
  const int64_t p0 = s_off[0], p1 = max(s_off[0], s_off[nb]);
  for (int64_t p = p0 + threadIdx.x; p < p1; p += blockDim.x) {
    int lo = 0, hi = nb;  // s_off[lo] <= p < s_off[hi] (for non-decreasing offsets)
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_off[mid] <= p) lo = mid;
      else hi = mid;
    }
    const uint32_t rel = static_cast<uint32_t>(r0 + lo);
    const int t = static_cast<int>(t0 + rel / B32);
    const uint32_t b = rel % B32;
    const int64_t rb = __ldg(a.roff + t);
    const int64_t E = __ldg(a.roff + t + 1) - rb;
    const int64_t id = ld_int<IT>(a.indices, p);
    uint32_t key;
    if (id >= 0 && id < E) {
      key = static_cast<uint32_t>(rb + id);
    } else {
      key = a.sentinel;
      ++bad;
    }
    a.keys[p] = key;
    a.vals[p] = b;
    if (PSW) a.psw_out[p] = __ldg(a.psw + p);
  }
  if (bad) atomicAdd(&s_bad, bad);
  __syncthreads();
  if (threadIdx.x == 0) stat_add(a.stats, TBE_STAT_UNREPAIRED, s_bad);
}

// ------------------------------------------------------------------------------------------
// radix sort
// ------------------------------------------------------------------------------------------
// The contiguous range of positions owned by CTA c of G: whole tiles, balanced.
__device__ __forceinline__ void segment_of(int64_t N, int c, int G, int64_t* b0, int64_t* b1) {
  const int64_t nt = (N + kSortTile - 1) / kSortTile;
  const int64_t t0 = nt * c / G, t1 = nt * (c + 1) / G;
  *b0 = min(N, t0 * kSortTile);
  *b1 = min(N, t1 * kSortTile);
}

__global__ void __launch_bounds__(kThreads) radix_upsweep_kernel(const uint32_t* keys,
                                                                const uint32_t* counters, int shift,
                                                                uint32_t* counts, int G) {
  __shared__ uint32_t hist[kThreads / kWarp][kRadix];
  const int w = threadIdx.x / kWarp;
  for (int j = threadIdx.x; j < (kThreads / kWarp) * kRadix; j += blockDim.x) (&hist[0][0])[j] = 0;
  __syncthreads();
  int64_t b0, b1;
  segment_of(counters[TBE_CNT_N], blockIdx.x, G, &b0, &b1);
  // b0 is a multiple of the tile (16-byte aligned); vector loads for the bulk
  const int64_t nvec = (b1 - b0) / 4;
  const uint4* kv = reinterpret_cast<const uint4*>(keys + b0);
  for (int64_t i = threadIdx.x; i < nvec; i += blockDim.x) {
    const uint4 k = kv[i];
    atomicAdd(&hist[w][(k.x >> shift) & (kRadix - 1)], 1u);
    atomicAdd(&hist[w][(k.y >> shift) & (kRadix - 1)], 1u);
    atomicAdd(&hist[w][(k.z >> shift) & (kRadix - 1)], 1u);
    atomicAdd(&hist[w][(k.w >> shift) & (kRadix - 1)], 1u);
  }
  for (int64_t i = b0 + nvec * 4 + threadIdx.x; i < b1; i += blockDim.x)
    atomicAdd(&hist[w][(keys[i] >> shift) & (kRadix - 1)], 1u);
  __syncthreads();
  for (int d = threadIdx.x; d < kRadix; d += blockDim.x) {
    uint32_t s = 0;
    for (int k = 0; k < kThreads / kWarp; ++k) s += hist[k][d];
    counts[static_cast<int64_t>(d) * G + blockIdx.x] = s;
  }
}

// Exclusive scan, in place, of n counters (one CTA of 1024 threads; n <= 256 * 1024).
__global__ void __launch_bounds__(1024) exclusive_scan_kernel(uint32_t* data, int n) {
  __shared__ uint32_t warp_tot[32];
  const int per = (n + blockDim.x - 1) / blockDim.x;
  const int beg = min(n, static_cast<int>(threadIdx.x) * per), end = min(n, beg + per);
  uint32_t local = 0;
  for (int i = beg; i < end; ++i) local += data[i];
  // block exclusive scan of `local`
  const int lane = lane_id(), w = threadIdx.x / kWarp;
  uint32_t v = local;
  for (int d = 1; d < kWarp; d <<= 1) {
    const uint32_t o = __shfl_up_sync(FULL, v, d);
    if (lane >= d) v += o;
  }
  if (lane == kWarp - 1) warp_tot[w] = v;
  __syncthreads();
  if (w == 0) {
    uint32_t x = lane < static_cast<int>(blockDim.x / kWarp) ? warp_tot[lane] : 0;
    for (int d = 1; d < kWarp; d <<= 1) {
      const uint32_t o = __shfl_up_sync(FULL, x, d);
      if (lane >= d) x += o;
    }
    warp_tot[lane] = x;  // inclusive over warps
  }
  __syncthreads();
  uint32_t run = v - local + (w > 0 ? warp_tot[w - 1] : 0);
  for (int i = beg; i < end; ++i) {
    const uint32_t c = data[i];
    data[i] = run;
    run += c;
  }
}

template <bool PSW>
__global__ void __launch_bounds__(kThreads) radix_downsweep_kernel(
    const uint32_t* keys_in, const uint32_t* vals_in, const float* psw_in, uint32_t* keys_out,
    uint32_t* vals_out, float* psw_out, const uint32_t* counters, const uint32_t* scanned,
    int shift, int G) {
  extern __shared__ __align__(16) uint32_t s_dyn[];
  uint32_t* s_keys = s_dyn;
  uint32_t* s_vals = s_dyn + kSortTile;
  float* s_psw = reinterpret_cast<float*>(s_dyn + 2 * kSortTile);
  __shared__ uint32_t s_whist[kThreads / kWarp][kRadix];
  __shared__ uint32_t s_run[kRadix];
  __shared__ uint32_t s_dstart[kRadix];
  __shared__ uint32_t s_tcount[kRadix];
  __shared__ uint32_t s_wsum[kThreads / kWarp];

  const int lane = lane_id(), w = threadIdx.x / kWarp;
  const unsigned lt = lanemask_lt();
  int64_t b0, b1;
  segment_of(counters[TBE_CNT_N], blockIdx.x, G, &b0, &b1);
  for (int d = threadIdx.x; d < kRadix; d += blockDim.x)
    s_run[d] = scanned[static_cast<int64_t>(d) * G + blockIdx.x];

  for (int64_t tb = b0; tb < b1; tb += kSortTile) {
    const int n = static_cast<int>(min(static_cast<int64_t>(kSortTile), b1 - tb));
    for (int j = threadIdx.x; j < (kThreads / kWarp) * kRadix; j += blockDim.x) (&s_whist[0][0])[j] = 0;
    __syncthreads();

    uint32_t k[kSortItems], v[kSortItems], rank[kSortItems];
    float pw[kSortItems];
#pragma unroll
    for (int i = 0; i < kSortItems; ++i) {
      const int e = w * (kSortItems * kWarp) + i * kWarp + lane;
      if (e < n) {
        k[i] = keys_in[tb + e];
        v[i] = vals_in[tb + e];
        if (PSW) pw[i] = psw_in[tb + e];
      } else {
        k[i] = 0;
        v[i] = 0;
        pw[i] = 0.f;
      }
    }
#pragma unroll
    for (int i = 0; i < kSortItems; ++i) {
      const int e = w * (kSortItems * kWarp) + i * kWarp + lane;
      const uint32_t d = e < n ? ((k[i] >> shift) & (kRadix - 1)) : static_cast<uint32_t>(kRadix);
      const unsigned peers = __match_any_sync(FULL, d);
      const int leader = __ffs(peers) - 1;
      uint32_t base = 0;
      if (lane == leader && d < kRadix) {
        base = s_whist[w][d];
        s_whist[w][d] = base + __popc(peers);
      }
      base = __shfl_sync(FULL, base, leader);
      rank[i] = base + __popc(peers & lt);
      __syncwarp();
    }
    __syncthreads();
    // per digit: exclusive prefix over warps, tile count
    for (int d = threadIdx.x; d < kRadix; d += blockDim.x) {
      uint32_t s = 0;
#pragma unroll
      for (int q = 0; q < kThreads / kWarp; ++q) {
        const uint32_t c = s_whist[q][d];
        s_whist[q][d] = s;
        s += c;
      }
      s_tcount[d] = s;
    }
    __syncthreads();
    // exclusive scan of tile counts over digits (kRadix == kThreads: one digit per thread)
    {
      const uint32_t c = s_tcount[threadIdx.x];
      uint32_t x = c;
      for (int d = 1; d < kWarp; d <<= 1) {
        const uint32_t o = __shfl_up_sync(FULL, x, d);
        if (lane >= d) x += o;
      }
      if (lane == kWarp - 1) s_wsum[w] = x;
      __syncthreads();
      uint32_t before = 0;
      for (int q = 0; q < w; ++q) before += s_wsum[q];
      s_dstart[threadIdx.x] = before + x - c;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kSortItems; ++i) {
      const int e = w * (kSortItems * kWarp) + i * kWarp + lane;
      if (e < n) {
        const uint32_t d = (k[i] >> shift) & (kRadix - 1);
        const uint32_t pos = s_dstart[d] + s_whist[w][d] + rank[i];
        s_keys[pos] = k[i];
        s_vals[pos] = v[i];
        if (PSW) s_psw[pos] = pw[i];
      }
    }
    __syncthreads();
    for (int j = threadIdx.x; j < n; j += blockDim.x) {
      const uint32_t key = s_keys[j];
      const uint32_t d = (key >> shift) & (kRadix - 1);
      const uint32_t g = s_run[d] + (static_cast<uint32_t>(j) - s_dstart[d]);
      keys_out[g] = key;
      vals_out[g] = s_vals[j];
      if (PSW) psw_out[g] = s_psw[j];
    }
    __syncthreads();
    for (int d = threadIdx.x; d < kRadix; d += blockDim.x) s_run[d] += s_tcount[d];
    __syncthreads();
  }
}

// ------------------------------------------------------------------------------------------
// run-length encoding
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ void rle_segment(int64_t N, int c, int G, int64_t* b0, int64_t* b1) {
  const int64_t per = (N + G - 1) / G;
  *b0 = min(N, per * c);
  *b1 = min(N, *b0 + per);
}

__device__ __forceinline__ uint32_t block_sum_u32(uint32_t v, uint32_t* sh) {
  const int lane = lane_id(), w = threadIdx.x / kWarp;
  for (int m = 16; m > 0; m >>= 1) v += __shfl_xor_sync(FULL, v, m);
  __syncthreads();
  if (lane == 0) sh[w] = v;
  __syncthreads();
  uint32_t r = 0;
  for (int i = 0; i < static_cast<int>(blockDim.x / kWarp); ++i) r += sh[i];
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(kThreads) rle_count_kernel(const uint32_t* keys,
                                                            const uint32_t* counters,
                                                            uint32_t* rle_counts, int G) {
  __shared__ uint32_t sh[kThreads / kWarp];
  const int64_t N = counters[TBE_CNT_N];
  int64_t b0, b1;
  rle_segment(N, blockIdx.x, G, &b0, &b1);
  uint32_t heads = 0;
  for (int64_t i = b0 + threadIdx.x; i < b1; i += blockDim.x)
    heads += (i == 0 || keys[i] != keys[i - 1]) ? 1u : 0u;
  heads = block_sum_u32(heads, sh);
  if (threadIdx.x == 0) rle_counts[blockIdx.x] = heads;
}

__global__ void __launch_bounds__(kThreads) rle_write_kernel(const uint32_t* keys,
                                                            uint32_t* counters,
                                                            const uint32_t* rle_counts, int G,
                                                            uint32_t* unique, uint32_t* run_off,
                                                            uint32_t u_cap) {
  __shared__ uint32_t sh[kThreads / kWarp];
  __shared__ uint32_t s_wcnt[kThreads / kWarp];
  const int lane = lane_id(), w = threadIdx.x / kWarp;
  const int64_t N = counters[TBE_CNT_N];
  uint32_t before = 0;
  for (int c = threadIdx.x; c < static_cast<int>(blockIdx.x); c += blockDim.x) before += rle_counts[c];
  uint32_t base = block_sum_u32(before, sh);
  int64_t b0, b1;
  rle_segment(N, blockIdx.x, G, &b0, &b1);
  for (int64_t tb = b0; tb < b1; tb += blockDim.x) {
    const int64_t i = tb + threadIdx.x;
    bool head = false;
    uint32_t key = 0;
    if (i < b1) {
      key = keys[i];
      head = (i == 0) || key != keys[i - 1];
    }
    const unsigned bal = __ballot_sync(FULL, head);
    if (lane == 0) s_wcnt[w] = __popc(bal);
    __syncthreads();
    uint32_t pre = 0, tot = 0;
    for (int q = 0; q < static_cast<int>(blockDim.x / kWarp); ++q) {
      if (q < w) pre += s_wcnt[q];
      tot += s_wcnt[q];
    }
    if (head) {
      const uint32_t r = base + pre + __popc(bal & lanemask_lt());
      if (r < u_cap) {
        unique[r] = key;
        run_off[r] = static_cast<uint32_t>(i);
      }
    }
    base += tot;
    __syncthreads();
  }
  if (blockIdx.x == gridDim.x - 1 && threadIdx.x == 0) {
    counters[TBE_CNT_RUNS] = base;
    if (base <= u_cap) run_off[base] = static_cast<uint32_t>(N);
  }
}

}  // namespace

cudaError_t launch_expand(const Problem& P, const BwdCtx& c, cudaStream_t s) {
  ExpandArgs a;
  a.indices = c.indices;
  a.offsets = c.offsets;
  a.psw = c.psw;
  a.roff = c.roff;
  a.B = c.B;
  a.TB = c.TB;
  a.num_indices = c.num_indices;
  a.sentinel = static_cast<uint32_t>(c.total_rows);
  a.keys = c.keys[0];
  a.vals = c.vals[0];
  a.psw_out = c.pswbuf[0];
  a.counters = c.counters;
  a.stats = c.stats;
  const int64_t grid64 = (c.TB + kExpandBags - 1) / kExpandBags;
  const int grid = static_cast<int>(grid64 < 1 ? 1 : grid64);
  const bool psw = P.weighted;
  if (P.itype == TBE_I32) {
    if (psw) expand_kernel<int32_t, true><<<grid, kThreads, 0, s>>>(a);
    else expand_kernel<int32_t, false><<<grid, kThreads, 0, s>>>(a);
  } else {
    if (psw) expand_kernel<int64_t, true><<<grid, kThreads, 0, s>>>(a);
    else expand_kernel<int64_t, false><<<grid, kThreads, 0, s>>>(a);
  }
  note_launch();  // a single CTA when there are no bags: it records the lookup count (0)
  return cudaGetLastError();
}

size_t sort_smem_bytes(bool psw) { return sizeof(uint32_t) * kSortTile * (psw ? 3 : 2); }

cudaError_t launch_sort(const Problem& P, const BwdCtx& c, const BwdLayout& L, cudaStream_t s) {
  const bool psw = P.weighted;
  const size_t smem = sort_smem_bytes(psw);
  // the opt-in shared memory size is a per-device function attribute: set it once per device
  static std::atomic<uint64_t> attr_set[2] = {{0}, {0}};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = uint64_t(1) << (dev & 63);
  if ((attr_set[psw ? 1 : 0].load() & bit) == 0) {
    e = psw ? cudaFuncSetAttribute(radix_downsweep_kernel<true>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)
            : cudaFuncSetAttribute(radix_downsweep_kernel<false>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_set[psw ? 1 : 0].fetch_or(bit);
  }
  const int G = L.sort_grid;
  int cur = 0;
  for (int pass = 0; pass < L.passes; ++pass) {
    const int shift = pass * kRadixBits;
    radix_upsweep_kernel<<<G, kThreads, 0, s>>>(c.keys[cur], c.counters, shift, c.sort_counts, G);
    note_launch();
    exclusive_scan_kernel<<<1, 1024, 0, s>>>(c.sort_counts, kRadix * G);
    note_launch();
    if (psw)
      radix_downsweep_kernel<true><<<G, kThreads, smem, s>>>(
          c.keys[cur], c.vals[cur], c.pswbuf[cur], c.keys[cur ^ 1], c.vals[cur ^ 1], c.pswbuf[cur ^ 1],
          c.counters, c.sort_counts, shift, G);
    else
      radix_downsweep_kernel<false><<<G, kThreads, smem, s>>>(
          c.keys[cur], c.vals[cur], nullptr, c.keys[cur ^ 1], c.vals[cur ^ 1], nullptr, c.counters,
          c.sort_counts, shift, G);
    note_launch();
    cur ^= 1;
  }
  return cudaGetLastError();
}

cudaError_t launch_rle(const Problem& P, const BwdCtx& c, const BwdLayout& L, cudaStream_t s) {
  (void)P;
  const uint32_t* keys = c.keys[L.final_buf];
  rle_count_kernel<<<L.rle_grid, kThreads, 0, s>>>(keys, c.counters, c.rle_counts, L.rle_grid);
  note_launch();
  rle_write_kernel<<<L.rle_grid, kThreads, 0, s>>>(keys, c.counters, c.rle_counts, L.rle_grid,
                                                   c.unique, c.run_off, c.u_cap);
  note_launch();
  return cudaGetLastError();
}

}  // namespace tbe
