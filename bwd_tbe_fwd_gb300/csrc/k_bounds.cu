// k_bounds.cu -- validation and repair of offsets and ids before the forward pass.
//
// "Modernizing Table Batched Embeddings with FBTriton", section 2 ("Bounds checking"): a
// validation step that repairs invalid input tensors, with offsets validated and repaired by
// a separate small kernel.  The pages do not state the repair rule; the rule implemented here:
//   offsets[T*B] is clamped into [0, num_indices]; offsets[0] becomes 0; every other offset is
//   clamped into [0, offsets[T*B]] and raised to the largest offset before it (a prefix
//   maximum), so bags never overlap and together cover [0, offsets[T*B]); then every id of
//   bag (t, b) outside [0, E[t]) becomes 0.
// Three launches: a per-segment maximum of the clamped inner offsets, the prefix-maximum
// repair of each segment (carrying the maxima of the segments before it), and the id check,
// which finds each lookup's table from the table starts offsets[t*B] kept in shared memory.
// Counts go to d_stats with one atomic per block.
#include "tbe_internal.cuh"

namespace tbe {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ int64_t block_reduce_max(int64_t v, int64_t* sh) {
  const int lane = lane_id(), w = threadIdx.x / kWarp;
  for (int m = 16; m > 0; m >>= 1) v = max(v, static_cast<int64_t>(__shfl_xor_sync(0xffffffffu, v, m)));
  __syncthreads();
  if (lane == 0) sh[w] = v;
  __syncthreads();
  int64_t r = sh[0];
  for (int i = 1; i < static_cast<int>(blockDim.x / kWarp); ++i) r = max(r, sh[i]);
  __syncthreads();
  return r;
}

__device__ __forceinline__ unsigned long long block_sum(unsigned long long v, unsigned long long* sh) {
  const int lane = lane_id(), w = threadIdx.x / kWarp;
  for (int m = 16; m > 0; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
  __syncthreads();
  if (lane == 0) sh[w] = v;
  __syncthreads();
  unsigned long long r = 0;
  for (int i = 0; i < static_cast<int>(blockDim.x / kWarp); ++i) r += sh[i];
  __syncthreads();
  return r;
}

// ws[0] = repaired last offset; ws[1 + c] = max of the clamped inner offsets of segment c.
template <typename IT>
__global__ void __launch_bounds__(kThreads) offsets_max_kernel(const IT* offsets, int64_t TB,
                                                              int64_t num_indices, int64_t* ws) {
  __shared__ int64_t sh[kThreads / kWarp];
  const int64_t last = clamp64(static_cast<int64_t>(offsets[TB]), 0, num_indices);
  const int64_t inner = TB > 1 ? TB - 1 : 0;  // offsets[1 .. TB-1]
  const int64_t seg = (inner + gridDim.x - 1) / gridDim.x;
  const int64_t i0 = 1 + seg * blockIdx.x, i1 = min(1 + inner, i0 + seg);
  int64_t m = 0;
#pragma unroll 8
  for (int64_t i = i0 + threadIdx.x; i < i1; i += blockDim.x)
    m = max(m, clamp64(static_cast<int64_t>(offsets[i]), 0, last));
  m = block_reduce_max(m, sh);
  if (threadIdx.x == 0) {
    ws[1 + blockIdx.x] = m;
    if (blockIdx.x == 0) ws[0] = last;
  }
}

// Each thread repairs kFixPerThread consecutive offsets per tile: a running maximum over its
// own offsets, then one block-wide scan of the threads' maxima (a tile of 2048 offsets per
// round of barriers rather than 256: the stress batch's 4.2M offsets take 4 rounds per CTA).
constexpr int kFixPerThread = 8;

template <typename IT>
__global__ void __launch_bounds__(kThreads) offsets_fix_kernel(IT* offsets, int64_t TB,
                                                              const int64_t* ws,
                                                              unsigned long long* stats) {
  constexpr int V = kFixPerThread;
  __shared__ int64_t sh[kThreads / kWarp];
  __shared__ unsigned long long shc[kThreads / kWarp];
  const int lane = lane_id(), w = threadIdx.x / kWarp;
  const int64_t last = ws[0];
  // carry-in: the largest clamped offset of the segments before this one (offsets[0] := 0)
  int64_t carry = 0;
  for (int c = threadIdx.x; c < static_cast<int>(blockIdx.x); c += blockDim.x) carry = max(carry, ws[1 + c]);
  carry = block_reduce_max(carry, sh);

  const int64_t inner = TB > 1 ? TB - 1 : 0;
  const int64_t seg = (inner + gridDim.x - 1) / gridDim.x;
  const int64_t i0 = 1 + seg * blockIdx.x, i1 = min(1 + inner, i0 + seg);
  unsigned long long changed = 0;
  for (int64_t base = i0; base < i1; base += static_cast<int64_t>(blockDim.x) * V) {  // block-uniform
    const int64_t ib = base + static_cast<int64_t>(threadIdx.x) * V;
    int64_t orig[V], v[V];
#pragma unroll
    for (int u = 0; u < V; ++u) orig[u] = ib + u < i1 ? static_cast<int64_t>(offsets[ib + u]) : 0;
    // inclusive prefix maximum over the thread's own offsets (clamped into [0, last]; a slot
    // past the segment holds 0, which changes no maximum)
    int64_t run = 0;
#pragma unroll
    for (int u = 0; u < V; ++u) {
      run = max(run, clamp64(orig[u], 0, last));
      v[u] = run;
    }
    // inclusive prefix maximum of the threads' maxima over the block
    int64_t x = run;
    for (int d = 1; d < kWarp; d <<= 1) {
      const int64_t o = __shfl_up_sync(0xffffffffu, x, d);
      if (lane >= d) x = max(x, o);
    }
    const int64_t x_prev = __shfl_up_sync(0xffffffffu, x, 1);
    __syncthreads();
    if (lane == kWarp - 1) sh[w] = x;
    __syncthreads();
    int64_t before = carry;  // the largest offset before this thread's first
    for (int k = 0; k < w; ++k) before = max(before, sh[k]);
    if (lane > 0) before = max(before, x_prev);
    int64_t tile_max = carry;
    for (int k = 0; k < static_cast<int>(blockDim.x / kWarp); ++k) tile_max = max(tile_max, sh[k]);
#pragma unroll
    for (int u = 0; u < V; ++u) {
      const int64_t f = max(v[u], before);
      if (ib + u < i1 && f != orig[u]) {
        offsets[ib + u] = static_cast<IT>(f);
        ++changed;
      }
    }
    carry = tile_max;
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    if (TB > 0 && static_cast<int64_t>(offsets[0]) != 0) {
      offsets[0] = IT(0);
      ++changed;
    }
    if (static_cast<int64_t>(offsets[TB]) != last) {
      offsets[TB] = static_cast<IT>(last);
      ++changed;
    }
  }
  changed = block_sum(changed, shc);
  if (threadIdx.x == 0) stat_add(stats, TBE_STAT_BAD_OFFSETS, changed);
}

// Every lookup p in [0, N): its table is the t with offsets[t*B] <= p < offsets[(t+1)*B].
// A thread checks 8 consecutive ids per step (two or four 16-byte loads), finds the table of
// the first by binary search over the table starts in shared memory and walks forward for the
// rest; the row counts of the tables sit in shared memory too.
template <typename IT>
__global__ void __launch_bounds__(kThreads) indices_fix_kernel(IT* indices, const IT* offsets,
                                                              int T, int64_t B,
                                                              const int64_t* roff,
                                                              const int64_t* ws,
                                                              unsigned long long* stats, int vec_ok) {
  extern __shared__ int32_t tshared[];  // [T+1] table starts, then [T] row counts (both < 2^31)
  int32_t* tstart = tshared;
  int32_t* trows = tshared + T + 1;
  __shared__ unsigned long long shc[kThreads / kWarp];
  const int64_t N = ws[0];
  for (int t = threadIdx.x; t <= T; t += blockDim.x)
    tstart[t] = static_cast<int32_t>(clamp64(static_cast<int64_t>(offsets[t * B]), 0, N));
  for (int t = threadIdx.x; t < T; t += blockDim.x) trows[t] = static_cast<int32_t>(__ldg(roff + t + 1) - __ldg(roff + t));
  __syncthreads();
  unsigned long long bad = 0;
  constexpr int V = 8;                                  // ids per thread per step
  constexpr int W = V * static_cast<int>(sizeof(IT)) / 16;  // 16-byte loads per step
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x * V;
  for (int64_t p0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * V; p0 < N; p0 += stride) {
    IT id[V];
    if (vec_ok && p0 + V <= N) {
      const uint4* src = reinterpret_cast<const uint4*>(indices + p0);
#pragma unroll
      for (int w = 0; w < W; ++w) {
        const uint4 r = src[w];
        const uint32_t words[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) reinterpret_cast<uint32_t*>(id)[w * 4 + q] = words[q];
      }
    } else {
#pragma unroll
      for (int u = 0; u < V; ++u) id[u] = p0 + u < N ? indices[p0 + u] : IT(0);
    }
    int lo = 0, hi = T;  // tstart[lo] <= p0 < tstart[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (tstart[mid] <= p0) lo = mid;
      else hi = mid;
    }
#pragma unroll
    for (int u = 0; u < V; ++u) {
      const int64_t p = p0 + u;
      if (p >= N) break;
      while (lo + 1 < T && tstart[lo + 1] <= p) ++lo;  // next table (tables can be empty)
      const int64_t v = static_cast<int64_t>(id[u]);
      if (v < 0 || v >= trows[lo]) {
        indices[p] = IT(0);
        ++bad;
      }
    }
  }
  bad = block_sum(bad, shc);
  if (threadIdx.x == 0) stat_add(stats, TBE_STAT_BAD_INDICES, bad);
}

template <typename IT>
cudaError_t launch_typed(const Problem& P, const tbe_tables& tab, void* indices, void* offsets,
                         int64_t* ws, int grid, unsigned long long* stats, bool with_ids, cudaStream_t s) {
  IT* off = static_cast<IT*>(offsets);
  offsets_max_kernel<IT><<<grid, kThreads, 0, s>>>(off, P.TB, P.num_indices, ws);
  note_launch();
  offsets_fix_kernel<IT><<<grid, kThreads, 0, s>>>(off, P.TB, ws, stats);
  note_launch();
  if (with_ids && P.num_indices > 0) {
    const size_t smem = sizeof(int32_t) * (2 * P.T + 1);
    const int64_t want = (P.num_indices + 8 * kThreads - 1) / (8 * kThreads);
    const int64_t cap = static_cast<int64_t>(grid) * 2;  // two waves of the bounds grid
    const int g = static_cast<int>(want < cap ? (want < 1 ? 1 : want) : cap);
    indices_fix_kernel<IT><<<g, kThreads, smem, s>>>(static_cast<IT*>(indices), off, P.T, P.B,
                                                     tab.row_offsets, ws, stats,
                                                     reinterpret_cast<uintptr_t>(indices) % 16 == 0 ? 1 : 0);
    note_launch();
  }
  return cudaGetLastError();
}

}  // namespace

int bounds_grid(const DeviceInfo& dev) { return dev.sms * 4 < 1024 ? dev.sms * 4 : 1024; }

cudaError_t launch_bounds(const Problem& P, const tbe_tables& tab, void* indices, void* offsets,
                          int64_t* ws, int grid, unsigned long long* stats, bool with_ids, cudaStream_t s) {
  if (P.itype == TBE_I32) return launch_typed<int32_t>(P, tab, indices, offsets, ws, grid, stats, with_ids, s);
  return launch_typed<int64_t>(P, tab, indices, offsets, ws, grid, stats, with_ids, s);
}

}  // namespace tbe
