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
//   expand      one CTA per 32-512 consecutive bags (about 16K lookups from the mean bag length);
//               their lookups are one contiguous range, read
//               coalesced; each lookup finds its bag by binary search over the CTA's offsets in
//               shared memory and writes key = row_offsets[t] + id (uint32) and its bag b
//               (plus its per-sample weight when weighted).
//   radix sort  LSD, digits of 8 to 10 bits, as few passes as the key range allows
//               (ceil(bits/10), the range being sum E + 1 for an out-of-range sentinel), the
//               narrower digits first.  Each pass is
//               reduce-then-scan: a per-CTA digit histogram over a contiguous segment, one
//               exclusive scan of the [digit][CTA] counts, and a stable scatter in which each
//               CTA walks its segment in 4096-key tiles, ranks keys with warp-level match
//               (__match_any_sync; one ballot per digit bit in the first pass, whose digits
//               are mostly distinct) and per-warp digit counters in shared memory, reorders the
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
  int bags_per_cta;   // <= kExpandBags
  uint32_t* keys;
  uint32_t* vals;
  float* psw_out;
  uint32_t* counters;
  unsigned long long* stats;
  float* inv_len;              // NULL, or [TB]: 1 / L of each bag (unweighted mean pooling)
  int mean;                    // mean pooling: the factor is psw / L (1 / L unweighted)
  int nhist;                   // tables whose lookups stay out of the sort
  int hist_t[kMaxHistTables];  // ascending
};

template <typename IT, bool PSW>
__global__ void __launch_bounds__(kThreads) expand_kernel(ExpandArgs a) {
  __shared__ int64_t s_off[kExpandBags + 1];
  __shared__ uint32_t s_b[kExpandBags], s_rb[kExpandBags], s_E[kExpandBags], s_shift[kExpandBags];
  __shared__ unsigned long long s_bad;
  __shared__ int64_t s_hlen[kMaxHistTables];
  const int64_t N = clamp64(ld_int<IT>(a.offsets, a.TB), 0, a.num_indices);
  const int64_t i0 = static_cast<int64_t>(blockIdx.x) * a.bags_per_cta;
  const int nb = static_cast<int>(min(static_cast<int64_t>(a.bags_per_cta), a.TB - i0));
  // Lookups of the counts-path tables are left out: a lookup of table t lands at its position
  // minus the lookups of the counts-path tables before t, and N shrinks by all of them.
  if (threadIdx.x < a.nhist) {
    const int64_t h0 = a.hist_t[threadIdx.x] * a.B;
    const int64_t hs = clamp64(ld_int<IT>(a.offsets, h0), 0, N);
    s_hlen[threadIdx.x] = clamp64(ld_int<IT>(a.offsets, h0 + a.B), hs, N) - hs;
  }
  for (int k = threadIdx.x; k <= nb; k += blockDim.x) s_off[k] = clamp64(ld_int<IT>(a.offsets, i0 + k), 0, N);
  if (threadIdx.x == 0) s_bad = 0;
  __syncthreads();
  int64_t n_kept = N;
  for (int h = 0; h < a.nhist; ++h) n_kept -= s_hlen[h];
  if (threadIdx.x == 0 && blockIdx.x == 0) a.counters[TBE_CNT_N] = static_cast<uint32_t>(n_kept < 0 ? 0 : n_kept);
  unsigned long long bad = 0;
  if (threadIdx.x < nb && s_off[threadIdx.x + 1] < s_off[threadIdx.x]) ++bad;  // decreasing offsets
  for (int k = threadIdx.x + kThreads; k < nb; k += blockDim.x)
    if (s_off[k + 1] < s_off[k]) ++bad;
  const int64_t t0 = a.B > 0 ? i0 / a.B : 0;
  int64_t p0 = s_off[0], p1 = max(s_off[0], s_off[nb]);
  if (a.nhist > 0 && nb > 0 && a.B > 0 && t0 == (i0 + nb - 1) / a.B) {
    bool all = false;  // every bag of this CTA is in one counts-path table
    for (int h = 0; h < a.nhist; ++h) all |= a.hist_t[h] == t0;
    if (all) p1 = p0;
  }
  // per bag of the CTA: its bag index b, its table's first key and row count, and how far its
  // lookups move down (the counts-path lookups before its table); row count 0 marks a bag of a
  // counts-path table, whose lookups are left out
  for (int k = threadIdx.x; k < nb; k += blockDim.x) {
    const int64_t u = i0 + k;
    const int t = static_cast<int>(u / a.B);
    const int64_t rb = __ldg(a.roff + t);
    s_b[k] = static_cast<uint32_t>(u - static_cast<int64_t>(t) * a.B);
    s_rb[k] = static_cast<uint32_t>(rb);
    uint32_t E = static_cast<uint32_t>(__ldg(a.roff + t + 1) - rb);
    int64_t shift = 0;
    for (int h = 0; h < a.nhist; ++h) {
      if (a.hist_t[h] < t) shift += s_hlen[h];
      if (a.hist_t[h] == t) E = 0;
    }
    s_E[k] = E;
    s_shift[k] = static_cast<uint32_t>(shift);
    if (a.inv_len != nullptr) {  // the correctly rounded 1 / L of the bag's lookups, as psw / L with psw = 1
      const int64_t L = s_off[k + 1] - s_off[k];
      a.inv_len[u] = L > 0 ? __frcp_rn(static_cast<float>(L)) : 0.0f;
    }
  }
  __syncthreads();
  // Each thread takes a 4-aligned group of 4 consecutive lookups: 16- or 32-byte loads of
  // their ids (and psw), and, when no counts-path table moves lookups (each lands at its own
  // position), 16-byte stores of their keys, bags and factors.  Groups that straddle the CTA's
  // range or the buffers' alignment take scalar accesses.
  constexpr int U = 4;
  const int64_t pa = p0 & ~static_cast<int64_t>(U - 1);
  const bool in_place = a.nhist == 0;
  const bool vec_in = (reinterpret_cast<uintptr_t>(a.indices) & 15) == 0 &&
                      (!PSW || a.psw == nullptr || (reinterpret_cast<uintptr_t>(a.psw) & 15) == 0);
  for (int64_t pb = pa + static_cast<int64_t>(threadIdx.x) * U; pb < p1; pb += static_cast<int64_t>(U) * blockDim.x) {
    const bool whole = pb >= p0 && pb + U <= p1;
    int64_t id[U];
    float w[U];
    if (whole && vec_in) {
      if constexpr (sizeof(IT) == 8) {
        const longlong2* v = reinterpret_cast<const longlong2*>(static_cast<const IT*>(a.indices) + pb);
        const longlong2 x = __ldg(v), y = __ldg(v + 1);
        id[0] = x.x; id[1] = x.y; id[2] = y.x; id[3] = y.y;
      } else {
        const int4 x = __ldg(reinterpret_cast<const int4*>(static_cast<const IT*>(a.indices) + pb));
        id[0] = x.x; id[1] = x.y; id[2] = x.z; id[3] = x.w;
      }
      if (PSW) {
        if (a.psw != nullptr) {
          const float4 x = __ldg(reinterpret_cast<const float4*>(a.psw + pb));
          w[0] = x.x; w[1] = x.y; w[2] = x.z; w[3] = x.w;
        } else {
          w[0] = w[1] = w[2] = w[3] = 1.f;
        }
      }
    } else {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t p = pb + u;
        const bool in = p >= p0 && p < p1;
        id[u] = in ? ld_int<IT>(a.indices, p) : 0;
        if (PSW) w[u] = in ? (a.psw != nullptr ? __ldg(a.psw + p) : 1.f) : 0.f;
      }
    }
    const int64_t pf = pb < p0 ? p0 : pb;  // the group's first lookup of this CTA
    int lo = 0, hi = nb;  // s_off[lo] <= pf < s_off[hi] (for non-decreasing offsets)
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_off[mid] <= pf) lo = mid;
      else hi = mid;
    }
    uint32_t kk[U], vv[U];
    float ff[U];
    int64_t qq[U];  // where each lookup lands among the kept ones; -1: not this CTA's, or dropped
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t p = pb + u;
      kk[u] = 0;
      vv[u] = 0;
      ff[u] = 0.f;
      qq[u] = -1;
      if (p < p0 || p >= p1) continue;
      while (lo + 1 < nb && s_off[lo + 1] <= p) ++lo;  // the next bags (possibly empty ones)
      const uint32_t E = s_E[lo];
      const bool hist_bag = a.nhist > 0 && E == 0;
      const int64_t q = p - s_shift[lo];
      if (hist_bag || q < 0 || q >= n_kept) continue;  // (out of range only for unrepaired offsets)
      qq[u] = q;
      if (id[u] >= 0 && id[u] < static_cast<int64_t>(E)) {
        kk[u] = s_rb[lo] + static_cast<uint32_t>(id[u]);
      } else {
        kk[u] = a.sentinel;
        ++bad;
      }
      vv[u] = s_b[lo];
      // the lookup's factor: psw, over the bag length for mean pooling (correctly rounded)
      if (PSW) ff[u] = a.mean ? __fdiv_rn(w[u], static_cast<float>(s_off[lo + 1] - s_off[lo])) : w[u];
    }
    bool vec_out = whole && in_place;
#pragma unroll
    for (int u = 0; u < U; ++u) vec_out = vec_out && qq[u] == pb + u;
    if (vec_out) {  // one 16-byte store per array
      *reinterpret_cast<uint4*>(a.keys + pb) = make_uint4(kk[0], kk[1], kk[2], kk[3]);
      *reinterpret_cast<uint4*>(a.vals + pb) = make_uint4(vv[0], vv[1], vv[2], vv[3]);
      if (PSW) *reinterpret_cast<float4*>(a.psw_out + pb) = make_float4(ff[0], ff[1], ff[2], ff[3]);
    } else {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (qq[u] < 0) continue;
        a.keys[qq[u]] = kk[u];
        a.vals[qq[u]] = vv[u];
        if (PSW) a.psw_out[qq[u]] = ff[u];
      }
    }
  }
  if (bad) atomicAdd(&s_bad, bad);
  __syncthreads();
  if (threadIdx.x == 0) stat_add(a.stats, TBE_STAT_UNREPAIRED, s_bad);
}

// ------------------------------------------------------------------------------------------
// radix sort
// ------------------------------------------------------------------------------------------
constexpr int kWarpsPerBlock = kThreads / kWarp;

// The contiguous range of positions owned by CTA c of G: whole tiles, balanced.
__device__ __forceinline__ void segment_of(int64_t N, int c, int G, int64_t* b0, int64_t* b1) {
  const int64_t nt = (N + kSortTile - 1) / kSortTile;
  const int64_t t0 = nt * c / G, t1 = nt * (c + 1) / G;
  *b0 = min(N, t0 * kSortTile);
  *b1 = min(N, t1 * kSortTile);
}

// Per-CTA digit histogram of its segment -> counts[digit * G + c].
template <int RB>
__global__ void __launch_bounds__(kThreads) radix_upsweep_kernel(const uint32_t* keys,
                                                                const uint32_t* counters, int shift,
                                                                uint32_t* counts, int G) {
  constexpr int R = 1 << RB;
  __shared__ uint32_t hist[kWarpsPerBlock][R];
  const int w = threadIdx.x / kWarp;
  for (int j = threadIdx.x; j < kWarpsPerBlock * R; j += blockDim.x) (&hist[0][0])[j] = 0;
  __syncthreads();
  int64_t b0, b1;
  segment_of(counters[TBE_CNT_N], blockIdx.x, G, &b0, &b1);
  const int64_t nvec = (b1 - b0) / 4;  // b0 is a multiple of the tile: 16-byte aligned
  const uint4* kv = reinterpret_cast<const uint4*>(keys + b0);
  int64_t i = threadIdx.x;
  constexpr int UP = 4;  // 16-byte loads in flight per thread (2 or 8 measured slower)
  for (; i + (UP - 1) * static_cast<int64_t>(blockDim.x) < nvec; i += UP * blockDim.x) {
    uint4 k[UP];
#pragma unroll
    for (int u = 0; u < UP; ++u) k[u] = kv[i + u * blockDim.x];
#pragma unroll
    for (int u = 0; u < UP; ++u) {
      atomicAdd(&hist[w][(k[u].x >> shift) & (R - 1)], 1u);
      atomicAdd(&hist[w][(k[u].y >> shift) & (R - 1)], 1u);
      atomicAdd(&hist[w][(k[u].z >> shift) & (R - 1)], 1u);
      atomicAdd(&hist[w][(k[u].w >> shift) & (R - 1)], 1u);
    }
  }
  for (; i < nvec; i += blockDim.x) {
    const uint4 k0 = kv[i];
    atomicAdd(&hist[w][(k0.x >> shift) & (R - 1)], 1u);
    atomicAdd(&hist[w][(k0.y >> shift) & (R - 1)], 1u);
    atomicAdd(&hist[w][(k0.z >> shift) & (R - 1)], 1u);
    atomicAdd(&hist[w][(k0.w >> shift) & (R - 1)], 1u);
  }
  for (int64_t p = b0 + nvec * 4 + threadIdx.x; p < b1; p += blockDim.x)
    atomicAdd(&hist[w][(keys[p] >> shift) & (R - 1)], 1u);
  __syncthreads();
  for (int d = threadIdx.x; d < R; d += blockDim.x) {
    uint32_t s = 0;
#pragma unroll
    for (int k = 0; k < kWarpsPerBlock; ++k) s += hist[k][d];
    counts[static_cast<int64_t>(d) * G + blockIdx.x] = s;
  }
}

// Block-wide exclusive scan of one value per thread; returns the prefix, *total the sum.
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t* s_wsum, uint32_t* total) {
  const int lane = lane_id(), w = threadIdx.x / kWarp;
  uint32_t x = v;
  for (int d = 1; d < kWarp; d <<= 1) {
    const uint32_t o = __shfl_up_sync(FULL, x, d);
    if (lane >= d) x += o;
  }
  __syncthreads();
  if (lane == kWarp - 1) s_wsum[w] = x;
  __syncthreads();
  uint32_t before = 0, tot = 0;
  for (int q = 0; q < static_cast<int>(blockDim.x / kWarp); ++q) {
    const uint32_t c = s_wsum[q];
    if (q < w) before += c;
    tot += c;
  }
  if (total) *total = tot;
  return before + x - v;
}

// One CTA per digit: exclusive scan, in place, of that digit's G per-CTA counts, and the
// digit's total.
__global__ void __launch_bounds__(kThreads) digit_scan_kernel(uint32_t* counts, uint32_t* totals, int G) {
  __shared__ uint32_t s_wsum[kWarpsPerBlock];
  uint32_t* row = counts + static_cast<int64_t>(blockIdx.x) * G;
  const int per = (G + blockDim.x - 1) / blockDim.x;  // G <= 1024: at most 4
  const int beg = min(G, static_cast<int>(threadIdx.x) * per), end = min(G, beg + per);
  uint32_t c[4] = {0, 0, 0, 0}, local = 0;
  for (int i = beg; i < end; ++i) {
    c[i - beg] = row[i];
    local += c[i - beg];
  }
  uint32_t total;
  uint32_t run = block_exclusive_scan(local, s_wsum, &total);
  for (int i = beg; i < end; ++i) {
    row[i] = run;
    run += c[i - beg];
  }
  if (threadIdx.x == 0) totals[blockIdx.x] = total;
}

size_t downsweep_smem_bytes(int rb, bool psw) {
  const size_t R = size_t(1) << rb;
  return 2 * sizeof(uint32_t) * kSortTile * (psw ? 3 : 2) + sizeof(uint16_t) * kWarpsPerBlock * R +
         sizeof(uint32_t) * 3 * R;
}

constexpr uint32_t kTileWaitLimit = 1u << 22;

// Stable scatter of each CTA's segment, tile by tile, to its digits' output ranges.  A tile's
// keys, bags (and psw) arrive in shared memory by bulk copies (cp.async.bulk with an mbarrier)
// issued one tile ahead into the other of two buffers, so the copy engine streams the segment
// while the CTA ranks and scatters the current tile; the buffer that brought a tile in is then
// reused for its reordering.  A partial tile whose size is not a multiple of 16 bytes (only the
// last one of the whole array) is read with plain loads.
template <int RB, bool PSW>
__global__ void __launch_bounds__(kThreads, 2) radix_downsweep_kernel(
    const uint32_t* keys_in, const uint32_t* vals_in, const float* psw_in, uint32_t* keys_out,
    uint32_t* vals_out, float* psw_out, const uint32_t* counters, const uint32_t* scanned,
    const uint32_t* totals, int shift, int G, unsigned long long* stats) {
  constexpr int R = 1 << RB;
  constexpr int DPT = R / kThreads;  // digits per thread
  constexpr int NA = PSW ? 3 : 2;    // arrays per tile buffer
  extern __shared__ __align__(128) uint32_t s_dyn[];
  uint16_t* s_whist = reinterpret_cast<uint16_t*>(s_dyn + 2 * NA * kSortTile);  // [warps][R]
  uint32_t* s_run = reinterpret_cast<uint32_t*>(s_whist + kWarpsPerBlock * R);
  uint32_t* s_dstart = s_run + R;
  uint32_t* s_tcount = s_dstart + R;
  __shared__ uint32_t s_wsum[kWarpsPerBlock];
  __shared__ __align__(8) uint64_t s_bar[2];
  __shared__ int s_bulk[2];

  const int lane = lane_id(), w = threadIdx.x / kWarp;
  const unsigned lt = lanemask_lt();
  const int64_t N = counters[TBE_CNT_N];
  int64_t b0, b1;
  segment_of(N, blockIdx.x, G, &b0, &b1);
  {
    // output base of each digit for this CTA: exclusive prefix over the digit totals plus the
    // CTA's prefix within the digit
    uint32_t tt[DPT], tsum = 0;
#pragma unroll
    for (int q = 0; q < DPT; ++q) {
      tt[q] = totals[threadIdx.x * DPT + q];
      tsum += tt[q];
    }
    uint32_t run = block_exclusive_scan(tsum, s_wsum, nullptr);
#pragma unroll
    for (int q = 0; q < DPT; ++q) {
      const int d = threadIdx.x * DPT + q;
      s_run[d] = run + scanned[static_cast<int64_t>(d) * G + blockIdx.x];
      run += tt[q];
    }
  }
  // bulk-copy tile tb into buffer b (thread 0); false when its byte count is not a multiple of 16
  auto issue = [&](int64_t tb, int b) -> int {
    const uint32_t bytes = static_cast<uint32_t>(min(static_cast<int64_t>(kSortTile), b1 - tb)) * 4u;
    if (bytes % 16 != 0) return 0;
    uint32_t* dst = s_dyn + b * NA * kSortTile;
    mbar_arrive_expect_tx(&s_bar[b], bytes * NA);
    bulk_copy_g2s(dst, keys_in + tb, bytes, &s_bar[b]);
    bulk_copy_g2s(dst + kSortTile, vals_in + tb, bytes, &s_bar[b]);
    if (PSW) bulk_copy_g2s(dst + 2 * kSortTile, psw_in + tb, bytes, &s_bar[b]);
    return 1;
  };
  if (threadIdx.x == 0) {
    mbar_init(&s_bar[0], 1);
    mbar_init(&s_bar[1], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    s_bulk[0] = b0 < b1 ? issue(b0, 0) : 0;
  }
  __syncthreads();
  uint32_t phase[2] = {0u, 0u};
  bool failed = false;

  int cur = 0;
  for (int64_t tb = b0; tb < b1; tb += kSortTile, cur ^= 1) {
    const int n = static_cast<int>(min(static_cast<int64_t>(kSortTile), b1 - tb));
    // the next tile into the other buffer (free since the end of the previous tile)
    if (threadIdx.x == 0) s_bulk[cur ^ 1] = tb + kSortTile < b1 ? issue(tb + kSortTile, cur ^ 1) : 0;
    uint32_t* wh32 = reinterpret_cast<uint32_t*>(s_whist);
    for (int j = threadIdx.x; j < kWarpsPerBlock * R / 2; j += blockDim.x) wh32[j] = 0;
    uint32_t* s_keys = s_dyn + cur * NA * kSortTile;
    uint32_t* s_vals = s_keys + kSortTile;
    float* s_psw = reinterpret_cast<float*>(s_keys + 2 * kSortTile);
    const bool bulk = s_bulk[cur] != 0;
    if (bulk) {
      if (!mbar_wait_bounded(&s_bar[cur], phase[cur], kTileWaitLimit)) {
        failed = true;
        if (threadIdx.x == 0) stat_add(stats, TBE_STAT_WAIT_TIMEOUT, 1);
      }
      phase[cur] ^= 1u;
    }
    __syncthreads();

    uint32_t k[kSortItems], v[kSortItems], rank[kSortItems];
    float pw[kSortItems];
#pragma unroll
    for (int i = 0; i < kSortItems; ++i) {
      const int e = w * (kSortItems * kWarp) + i * kWarp + lane;
      const bool ok = e < n;
      if (bulk) {
        k[i] = ok ? s_keys[e] : 0u;
        v[i] = ok ? s_vals[e] : 0u;
        if (PSW) pw[i] = ok ? s_psw[e] : 0.f;
      } else {
        k[i] = ok ? keys_in[tb + e] : 0u;
        v[i] = ok ? vals_in[tb + e] : 0u;
        if (PSW) pw[i] = ok ? psw_in[tb + e] : 0.f;
      }
    }
    uint16_t* my_hist = s_whist + w * R;
#pragma unroll
    for (int i = 0; i < kSortItems; ++i) {
      const int e = w * (kSortItems * kWarp) + i * kWarp + lane;
      const uint32_t d = e < n ? ((k[i] >> shift) & (R - 1)) : static_cast<uint32_t>(R);
      // The lanes with the same digit.  The first pass reads the batch order, where a warp's 32
      // digits are mostly distinct: there one ballot per digit bit is cheaper than the match,
      // whose cost grows with the number of distinct values (it wins on the later passes, whose
      // input is grouped by the lower digits).
      unsigned peers;
      if (!PSW && shift == 0) {
        peers = __ballot_sync(FULL, d < R);
#pragma unroll
        for (int b = 0; b < RB; ++b) {
          const unsigned bb = __ballot_sync(FULL, (d >> b) & 1u);
          peers &= ((d >> b) & 1u) ? bb : ~bb;
        }
        if (d >= R) peers = 1u << lane;  // past the tile: no counter, no rank
      } else {
        peers = __match_any_sync(FULL, d);
      }
      const int leader = __ffs(peers) - 1;
      uint32_t base = 0;
      if (lane == leader && d < R) {
        base = my_hist[d];
        my_hist[d] = static_cast<uint16_t>(base + __popc(peers));
      }
      base = __shfl_sync(FULL, base, leader);
      rank[i] = base + __popc(peers & lt);
      __syncwarp();
    }
    __syncthreads();  // also: every thread has read its items out of the buffer
    // per digit: exclusive prefix over the warps (in place) and the tile count, then the
    // exclusive scan of the tile counts over the digits
    uint32_t tc[DPT], tsum = 0;
#pragma unroll
    for (int q = 0; q < DPT; ++q) {
      const int d = threadIdx.x * DPT + q;
      uint32_t sacc = 0;
#pragma unroll
      for (int w2 = 0; w2 < kWarpsPerBlock; ++w2) {
        const uint32_t c = s_whist[w2 * R + d];
        s_whist[w2 * R + d] = static_cast<uint16_t>(sacc);
        sacc += c;
      }
      tc[q] = sacc;
      tsum += sacc;
    }
    uint32_t run = block_exclusive_scan(tsum, s_wsum, nullptr);
#pragma unroll
    for (int q = 0; q < DPT; ++q) {
      const int d = threadIdx.x * DPT + q;
      s_dstart[d] = run;
      s_tcount[d] = tc[q];
      // each warp's base for the digit becomes its tile position (one lookup per item below)
#pragma unroll
      for (int w2 = 0; w2 < kWarpsPerBlock; ++w2)
        s_whist[w2 * R + d] = static_cast<uint16_t>(s_whist[w2 * R + d] + run);
      run += tc[q];
    }
    __syncthreads();
    // the reordered tile as (key, bag) pairs over the keys and bags of the buffer: one 8-byte
    // store per item at its scattered position (digit-indexed shared-memory accesses of a
    // tile in batch order are where the bank conflicts are), then conflict-free reads in order
    uint2* s_kv = reinterpret_cast<uint2*>(s_keys);
#pragma unroll
    for (int i = 0; i < kSortItems; ++i) {
      const int e = w * (kSortItems * kWarp) + i * kWarp + lane;
      if (e < n) {
        const uint32_t d = (k[i] >> shift) & (R - 1);
        const uint32_t pos = s_whist[w * R + d] + rank[i];
        s_kv[pos] = make_uint2(k[i], v[i]);
        if (PSW) s_psw[pos] = pw[i];
      }
    }
    __syncthreads();
    for (int j = threadIdx.x; j < n; j += blockDim.x) {
      const uint2 kv = s_kv[j];
      const uint32_t d = (kv.x >> shift) & (R - 1);
      const uint32_t g = s_run[d] + (static_cast<uint32_t>(j) - s_dstart[d]);
      if (!TBE_CHECK(g < N, stats)) continue;
      keys_out[g] = kv.x;
      vals_out[g] = kv.y;
      if (PSW) psw_out[g] = s_psw[j];
    }
    fence_proxy_async_smem();  // this buffer's generic accesses before the next bulk copy into it
    __syncthreads();
#pragma unroll
    for (int q = 0; q < DPT; ++q) {
      const int d = threadIdx.x * DPT + q;
      s_run[d] += s_tcount[d];
    }
    __syncthreads();
  }
  if (failed) {  // a copy that never signalled: wait once more (bounded) before the CTA exits
    mbar_wait_bounded(&s_bar[cur ^ 1], phase[cur ^ 1] ^ 1u, kTileWaitLimit);
  }
}

// ------------------------------------------------------------------------------------------
// run-length encoding: each thread owns 16 consecutive sorted keys of a 4096-key tile
// ------------------------------------------------------------------------------------------
constexpr int kRleItems = 16;
constexpr int kRleTile = kThreads * kRleItems;

__device__ __forceinline__ void rle_segment(int64_t N, int c, int G, int64_t* b0, int64_t* b1) {
  const int64_t nt = (N + kRleTile - 1) / kRleTile;
  *b0 = min(N, (nt * c / G) * kRleTile);
  *b1 = min(N, (nt * (c + 1) / G) * kRleTile);
}

// Loads keys[p0 .. p0+16) (clipped to n valid) and the key before p0; returns the head mask.
__device__ __forceinline__ uint32_t load_heads(const uint32_t* keys, int64_t p0, int64_t b1,
                                               uint32_t (&k)[kRleItems]) {
  const int64_t nvalid = b1 - p0;
  if (nvalid >= kRleItems) {
    const uint4* v = reinterpret_cast<const uint4*>(keys + p0);
#pragma unroll
    for (int q = 0; q < kRleItems / 4; ++q) {
      const uint4 x = v[q];
      k[4 * q] = x.x;
      k[4 * q + 1] = x.y;
      k[4 * q + 2] = x.z;
      k[4 * q + 3] = x.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < kRleItems; ++i) k[i] = i < nvalid ? keys[p0 + i] : 0u;
  }
  uint32_t prev = p0 > 0 ? keys[p0 - 1] : ~k[0];
  uint32_t mask = 0;
#pragma unroll
  for (int i = 0; i < kRleItems; ++i) {
    if (i < nvalid && k[i] != prev) mask |= 1u << i;
    prev = k[i];
  }
  return mask;
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
  __shared__ uint32_t sh[kWarpsPerBlock];
  const int64_t N = counters[TBE_CNT_N];
  int64_t b0, b1;
  rle_segment(N, blockIdx.x, G, &b0, &b1);
  uint32_t heads = 0;
  for (int64_t tb = b0; tb < b1; tb += kRleTile) {
    const int64_t p0 = tb + static_cast<int64_t>(threadIdx.x) * kRleItems;
    if (p0 < b1) {
      uint32_t k[kRleItems];
      heads += __popc(load_heads(keys, p0, b1, k));
    }
  }
  heads = block_sum_u32(heads, sh);
  if (threadIdx.x == 0) rle_counts[blockIdx.x] = heads;
}

__global__ void __launch_bounds__(kThreads) rle_write_kernel(const uint32_t* keys,
                                                            uint32_t* counters,
                                                            const uint32_t* rle_counts, int G,
                                                            uint32_t* unique, uint32_t* run_off,
                                                            uint32_t u_cap, unsigned long long* stats) {
  __shared__ uint32_t sh[kWarpsPerBlock];
  const int64_t N = counters[TBE_CNT_N];
  uint32_t before = 0;
  for (int c = threadIdx.x; c < static_cast<int>(blockIdx.x); c += blockDim.x) before += rle_counts[c];
  uint32_t base = block_sum_u32(before, sh);
  int64_t b0, b1;
  rle_segment(N, blockIdx.x, G, &b0, &b1);
  for (int64_t tb = b0; tb < b1; tb += kRleTile) {
    const int64_t p0 = tb + static_cast<int64_t>(threadIdx.x) * kRleItems;
    uint32_t k[kRleItems];
    const uint32_t mask = p0 < b1 ? load_heads(keys, p0, b1, k) : 0u;
    uint32_t total;
    uint32_t r = base + block_exclusive_scan(__popc(mask), sh, &total);
#pragma unroll
    for (int i = 0; i < kRleItems; ++i) {
      if (mask & (1u << i)) {
        if (TBE_GUARD(r < u_cap, stats)) {
          unique[r] = k[i];
          run_off[r] = static_cast<uint32_t>(p0 + i);
        }
        ++r;
      }
    }
    base += total;
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
  a.inv_len = c.inv_len;
  a.mean = P.pooling == TBE_POOL_MEAN;
  a.nhist = c.nhist;
  for (int h = 0; h < kMaxHistTables; ++h) a.hist_t[h] = h < c.nhist ? c.hist_t[h] : 0;
  // about 16K lookups per CTA: bags per CTA from the mean bag length the host can see
  const int64_t mean_len = c.TB > 0 ? (c.num_indices + c.TB - 1) / c.TB : 1;
  int bpc = kExpandBags;
  while (bpc > 32 && static_cast<int64_t>(bpc) * mean_len > 16384) bpc >>= 1;
  a.bags_per_cta = bpc;
  const int64_t grid64 = (c.TB + bpc - 1) / bpc;
  const int grid = static_cast<int>(grid64 < 1 ? 1 : grid64);
  const bool psw = P.scaled;
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

namespace {

// One LSD pass over digit [shift, shift + RB) of the keys in buffer `cur` into buffer cur ^ 1.
template <int RB>
cudaError_t sort_pass(const Problem& P, const BwdCtx& c, const BwdLayout& L, int cur, int shift, cudaStream_t s) {
  const bool psw = P.scaled;
  const size_t smem = downsweep_smem_bytes(RB, psw);
  // the opt-in shared memory size is a per-device function attribute: set it once per device
  static std::atomic<uint64_t> attr_set[2] = {{0}, {0}};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = uint64_t(1) << (dev & 63);
  if ((attr_set[psw ? 1 : 0].load() & bit) == 0) {
    e = psw ? cudaFuncSetAttribute(radix_downsweep_kernel<RB, true>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)
            : cudaFuncSetAttribute(radix_downsweep_kernel<RB, false>,
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    attr_set[psw ? 1 : 0].fetch_or(bit);
  }
  const int G = L.sort_grid;
  radix_upsweep_kernel<RB><<<G, kThreads, 0, s>>>(c.keys[cur], c.counters, shift, c.sort_counts, G);
  note_launch();
  digit_scan_kernel<<<1 << RB, kThreads, 0, s>>>(c.sort_counts, c.sort_totals, G);
  note_launch();
  if (psw)
    radix_downsweep_kernel<RB, true><<<G, kThreads, smem, s>>>(
        c.keys[cur], c.vals[cur], c.pswbuf[cur], c.keys[cur ^ 1], c.vals[cur ^ 1], c.pswbuf[cur ^ 1],
        c.counters, c.sort_counts, c.sort_totals, shift, G, c.stats);
  else
    radix_downsweep_kernel<RB, false><<<G, kThreads, smem, s>>>(
        c.keys[cur], c.vals[cur], nullptr, c.keys[cur ^ 1], c.vals[cur ^ 1], nullptr, c.counters,
        c.sort_counts, c.sort_totals, shift, G, c.stats);
  note_launch();
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_sort(const Problem& P, const BwdCtx& c, const BwdLayout& L, cudaStream_t s) {
  int cur = 0, shift = 0;
  for (int pass = 0; pass < L.passes; ++pass) {
    cudaError_t e;
    switch (L.pass_bits[pass]) {
      case 8: e = sort_pass<8>(P, c, L, cur, shift, s); break;
      case 9: e = sort_pass<9>(P, c, L, cur, shift, s); break;
      default: e = sort_pass<10>(P, c, L, cur, shift, s); break;
    }
    if (e != cudaSuccess) return e;
    shift += L.pass_bits[pass];
    cur ^= 1;
  }
  return cudaSuccess;
}

cudaError_t launch_rle(const Problem& P, const BwdCtx& c, const BwdLayout& L, cudaStream_t s) {
  (void)P;
  const uint32_t* keys = c.keys[L.final_buf];
  rle_count_kernel<<<L.rle_grid, kThreads, 0, s>>>(keys, c.counters, c.rle_counts, L.rle_grid);
  note_launch();
  rle_write_kernel<<<L.rle_grid, kThreads, 0, s>>>(keys, c.counters, c.rle_counts, L.rle_grid,
                                                   c.unique, c.run_off, c.u_cap, c.stats);
  note_launch();
  return cudaGetLastError();
}

}  // namespace tbe
