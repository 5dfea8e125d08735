// k_hist.cu -- the small-table forward as counts x table on the tcgen05 tensor cores.
//
// "Modernizing Table Batched Embeddings with FBTriton", section 2 ("The small-table histogram
// and tensor-core path"): for one feature with E <= 64 rows, 64 <= D <= 128, long bags (L >= 64),
// fp16 weights, fp32 output and no per-sample weights, a bag's pooled row is
//     out[b, :] = sum_e count[b, e] * W[e, :]
// where count[b, e] counts the bag's first 256 ids equal to e; ids after the 256th are added by a
// scalar path.  The pages evaluate counts x table with a Triton dot over 16 bags per program.
//
// GB300 design: a persistent CTA of 256 threads owns TMEM columns for one 128 x D fp32
// accumulator and keeps the table in shared memory as the B operand (written once, after the
// CTA's first tile's ids are counted).  Per tile of 128 bags:
//   1. the tile's 129 offsets go to shared memory; each warp streams the contiguous positions of
//      its 16 bags with four 16-byte id loads in flight per lane, walking the bag boundaries
//      forward, and for ids among the first 256 of their bag counts them with 32-bit
//      shared-memory atomics on packed 16-bit pairs (given a place to save them, the tile's
//      counts also go to global memory for the backward); the counts are then written as the
//      fp16 A tile (counts <= 256 are exact in fp16) in the canonical K-major layout without
//      swizzle (8 x 16-byte core matrices);
//   2. one thread issues four tcgen05.mma.cta_group::1.kind::f16 (M=128, N=D rounded up to 16,
//      K=16 each) and commits them to an mbarrier; the CTA waits on it (bounded);
//   3. all 8 warps read the accumulator (one bag per thread: warps w and w + 4 share TMEM lanes
//      32 (w % 4) .. + 31 and split the 32-column chunks) with tcgen05.ld 32x32b.x32, add the rows
//      of ids past the 256th, and store the pooled rows through shared memory as 128-byte pieces.
// Counts x table is exact up to fp32 rounding, so the result equals the gather's sum.
#include <atomic>

#include "tbe_internal.cuh"

namespace tbe {
namespace {

constexpr int kThreads = 256;       // 8 warps count; warps 0-3 (one bag per thread) read TMEM
constexpr int kM = 128;
constexpr int kK = 64;              // E padded to 64
constexpr int kMaxN = 128;          // D <= 128
constexpr int kHistIds = 256;       // ids per bag counted by the histogram
// id loads in flight per lane while counting: 16-byte loads in the forward, single ids in the
// backward (measured faster each way)
constexpr bool kFwdVecIds = true;
constexpr int kFwdLoads = 4;
constexpr bool kBwdVecIds = false;
constexpr int kBwdLoads = 16;
constexpr int kTileBytes = kM * kK * 2;  // A tile: 128 x 64 fp16 = 16 KB (B tile: 128 x 64 as well)
constexpr uint32_t kTmemCols = 128;
constexpr uint32_t kWaitLimit = 1u << 22;
constexpr unsigned FULL = 0xffffffffu;
// canonical K-major layout without swizzle: core matrices of 8 rows x 16 bytes; adjacent core
// matrices are 128 B apart along K (LBO) and 8 * 128 = 1024 B apart along M/N (SBO)
constexpr uint32_t kLBO = 128;
constexpr uint32_t kSBO = (kK / 8) * 128;

struct HistArgs {
  const __half* table;   // the table's rows (E x D), row-major
  const void* indices;
  const void* offsets;   // table-major offsets; this table's bags are offsets[t*B .. t*B+B]
  float* out;
  int64_t B;
  int64_t num_indices;
  int64_t bag0;          // t * B
  int E, D, N;           // N = D rounded up to a multiple of 16
  int col0, total_D;
  int fused_bounds;      // repair out-of-range ids in flight (row 0, written back) instead of skipping
  uint32_t* save_pairs;  // NULL, or [B][32]: each bag's count pairs, saved for the backward
  unsigned long long* stats;
};

__device__ __forceinline__ uint64_t smem_desc(uint32_t addr) {
  // start address, LBO and SBO in 16-byte units; bits 46-47 = 1 (descriptor version); no swizzle
  return static_cast<uint64_t>((addr >> 4) & 0x3FFF) | (static_cast<uint64_t>(kLBO >> 4) << 16) |
         (static_cast<uint64_t>(kSBO >> 4) << 32) | (uint64_t(1) << 46);
}

// kind::f16 instruction descriptor: fp32 accumulator, fp16 A and B, both K-major, shape M x N.
__device__ __forceinline__ uint32_t instr_desc(int M, int N) {
  return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// byte offset of element (row r, k) in a K-major tile
__device__ __forceinline__ uint32_t kmajor_offset(int r, int k) {
  return static_cast<uint32_t>((r >> 3) * kSBO + (k >> 3) * kLBO + (r & 7) * 16 + (k & 7) * 2);
}

__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t cols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(cols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t cols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols) : "memory");
}

__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n"
      "  .reg .pred p;\n"
      "  setp.ne.b32 p, %4, 0;\n"
      "  tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n"
      "}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive fp32 accumulator columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Offsets of a tile's bags made non-decreasing (a bag never ends before it starts): each entry
// becomes the running maximum of the ones before it.  Warp 0 scans the n + 1 <= 160 entries,
// five per lane; the caller synchronizes before and after.
__device__ __forceinline__ void monotone_offsets(int64_t* s_off, int n, int lane) {
  constexpr int kPer = 5;
  const int i0 = lane * kPer;
  int64_t v[kPer], m = INT64_MIN;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    if (i0 + j <= n) m = max(m, s_off[i0 + j]);
    v[j] = m;
  }
  int64_t incl = m;  // inclusive prefix maximum over the lanes
  for (int d = 1; d < kWarp; d <<= 1) {
    const int64_t o = __shfl_up_sync(FULL, incl, d);
    if (lane >= d) incl = max(incl, o);
  }
  int64_t before = __shfl_up_sync(FULL, incl, 1);
  if (lane == 0) before = INT64_MIN;
#pragma unroll
  for (int j = 0; j < kPer; ++j)
    if (i0 + j <= n) s_off[i0 + j] = max(v[j], before);
}

// Visits every lookup of the tile's bags once: warp w takes the bags [w * per, (w + 1) * per) of
// the tile, one contiguous range of positions, and streams it with U loads in flight per lane
// (16-byte loads of 16 / sizeof(IT) ids with VEC, else one id each); visit(r, bag, bag_start, id) gets the position relative to the
// tile's first lookup p0, the bag within the tile and that bag's first position.  The loads start
// at the 16-byte boundary at or below the range's first id (ids before it are loaded, not
// visited); one that would pass the range's end, or an ids array not 16-byte aligned, takes
// scalar loads.  A lane's positions only grow, so it walks its bag boundaries forward.
template <typename IT, bool VEC, int U, int kWarps, typename F>
__device__ __forceinline__ void for_each_lookup(const IT* ids, int64_t p0, bool vec_ok, const int* s_rel, int nb,
                                                int warp, int lane, F&& visit) {
  constexpr int V = VEC ? 16 / static_cast<int>(sizeof(IT)) : 1;
  vec_ok = vec_ok && VEC;
  const int per = (nb + kWarps - 1) / kWarps;
  const int bw0 = min(nb, warp * per), bw1 = min(nb, bw0 + per);
  const int r_beg = s_rel[bw0], r_end = s_rel[bw1];
  if (r_beg >= r_end) return;  // (so bw0 < bw1)
  int lo = bw0, cur = r_beg, nxt = s_rel[bw0 + 1];
  const int r_first = r_beg - static_cast<int>((p0 + r_beg) & (V - 1));  // 16-byte aligned
  for (int r0 = r_first; r0 < r_end; r0 += kWarp * V * U) {
    IT id[U][V];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int rv = r0 + (u * kWarp + lane) * V;
      if (vec_ok && rv + V <= r_end) {
        const uint4 x = __ldg(reinterpret_cast<const uint4*>(ids + rv));
        const IT* e = reinterpret_cast<const IT*>(&x);
#pragma unroll
        for (int j = 0; j < V; ++j) id[u][j] = e[j];
      } else {
#pragma unroll
        for (int j = 0; j < V; ++j) id[u][j] = (rv + j >= r_beg && rv + j < r_end) ? __ldg(ids + rv + j) : IT(0);
      }
    }
    bool past = false;
#pragma unroll
    for (int u = 0; u < U; ++u) {
#pragma unroll
      for (int j = 0; j < V; ++j) {
        const int r = r0 + (u * kWarp + lane) * V + j;
        past = past || r >= r_end;
        if (past || r < r_beg) continue;
        while (r >= nxt) {  // into the next bag (empty bags are stepped over)
          ++lo;
          cur = nxt;
          nxt = lo + 1 <= bw1 ? s_rel[lo + 1] : 0x7fffffff;
        }
        visit(r, lo, cur, id[u][j]);
      }
    }
  }
}

template <typename IT>
__global__ void __launch_bounds__(kThreads, 4) hist_tc_kernel(HistArgs a) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  // tiles 1024-byte aligned within the shared window (the launch adds 1 KB of slack)
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* a_tile = smem;                                   // 16 KB: counts as fp16
  uint8_t* b_tile = smem + kTileBytes;                      // 16 KB: the table
  uint32_t* pairs = reinterpret_cast<uint32_t*>(smem + 2 * kTileBytes);  // 16 KB: [128][32] count pairs
  __shared__ __align__(8) uint64_t mma_bar;
  __shared__ uint32_t s_tmem;
  __shared__ int s_failed;
  __shared__ int64_t s_off[kM + 1];
  __shared__ int s_rel[kM + 1];

  const int tid = threadIdx.x, lane = lane_id(), warp = tid / kWarp;
  const bool vec_ok = (reinterpret_cast<uintptr_t>(a.indices) & 15) == 0;  // 16-byte id loads
  const int64_t tiles = (a.B + kM - 1) / kM;

  // TMEM for the accumulator (warp 0 allocates for the CTA), the MMA completion barrier
  if (warp == 0) tmem_alloc(&s_tmem, kTmemCols);
  if (tid == 0) {
    mbar_init(&mma_bar, 1);
    s_failed = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const uint32_t idesc = instr_desc(kM, a.N);
  const uint64_t a_desc0 = smem_desc(smem_u32(a_tile)), b_desc0 = smem_desc(smem_u32(b_tile));
  uint32_t phase = 0;
  bool b_built = false;

  for (int64_t tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
    const int64_t b0 = tile * kM;
    // 1. histogram of the first 256 ids of each bag, straight into the fp16 A tile
    const int nb = static_cast<int>(min(static_cast<int64_t>(kM), a.B - b0));
    for (int i = tid; i < kM * kK / 2 / 4; i += kThreads) reinterpret_cast<uint4*>(pairs)[i] = make_uint4(0, 0, 0, 0);
    for (int i = tid; i <= kM; i += kThreads) {
      const int64_t o = clamp64(ld_int<IT>(a.offsets, a.bag0 + b0 + min(i, nb)), 0, a.num_indices);
      s_off[i] = o;
    }
    __syncthreads();
    if (warp == 0) monotone_offsets(s_off, nb, lane);  // guard: never let a bag end before it starts
    __syncthreads();
    {
      // positions relative to the tile's first lookup (32-bit), bag starts in shared memory
      const int64_t p0 = s_off[0];
      for (int i = tid; i <= nb; i += kThreads) s_rel[i] = static_cast<int>(s_off[i] - p0);
      __syncthreads();
      IT* ids = const_cast<IT*>(static_cast<const IT*>(a.indices)) + p0;
      uint32_t bad = 0;
      for_each_lookup<IT, kFwdVecIds, kFwdLoads, kThreads / kWarp>(ids, p0, vec_ok, s_rel, nb, warp, lane,
                                                           [&](int r, int lo, int cur, IT id) {
        if (static_cast<uint64_t>(static_cast<int64_t>(id)) >= static_cast<uint64_t>(a.E)) {
          ++bad;
          if (!a.fused_bounds) return;  // skipped (the scalar path skips it too)
          ids[r] = IT(0);  // repaired in flight: row 0, written back
          id = IT(0);
        }
        if (r - cur >= kHistIds) return;  // the scalar path adds it
        const uint32_t k = static_cast<uint32_t>(id);
        // two 16-bit counts per word (counts <= 256 never carry into the neighbour)
        atomicAdd(&pairs[lo * (kK / 2) + (k >> 1)], (k & 1u) << 16 | (~k & 1u));
      });
      if (bad) stat_add(a.stats, a.fused_bounds ? TBE_STAT_BAD_INDICES : TBE_STAT_UNREPAIRED, bad);
    }
    __syncthreads();
    if (a.save_pairs != nullptr)  // the tile's counts for a backward on the same batch
      for (int i = tid; i < nb * (kK / 8); i += kThreads)
        reinterpret_cast<uint4*>(a.save_pairs + b0 * (kK / 2))[i] = reinterpret_cast<const uint4*>(pairs)[i];
    if (!b_built) {
      // B tile (once per CTA, after its first tile's ids are counted, so that the id stream starts
      // at once and the CTAs' reads of the table from L2 spread out): element (n, k) = W[k][n] for
      // k < E and n < D, zero elsewhere.  A warp fills one 128-byte block (8 columns n x 8 rows k
      // of core matrix memory) per step, one 32-bit pair of rows (k, k + 1) of one column per
      // lane: the block covers every bank once
      for (int blk = warp; blk < (kMaxN / 8) * (kK / 8); blk += kThreads / kWarp) {
        const int n = (blk % (kMaxN / 8)) * 8 + (lane >> 2);
        const int k = (blk / (kMaxN / 8)) * 8 + (lane & 3) * 2;
        uint32_t w = 0;
        if (n < a.D) {
          const uint32_t h0 = k < a.E ? __half_as_ushort(a.table[static_cast<int64_t>(k) * a.D + n]) : 0u;
          const uint32_t h1 = k + 1 < a.E ? __half_as_ushort(a.table[static_cast<int64_t>(k + 1) * a.D + n]) : 0u;
          w = h0 | (h1 << 16);
        }
        *reinterpret_cast<uint32_t*>(b_tile + kmajor_offset(n, k)) = w;
      }
      b_built = true;
    }
    // counts -> fp16 A tile (exact: counts <= 256), 8 counts (one 16-byte row of a core matrix)
    // per item
    for (int q = tid; q < kM * (kK / 8); q += kThreads) {
      const int m = q / (kK / 8), kb = (q % (kK / 8)) * 8;
      const uint4 c = *reinterpret_cast<const uint4*>(&pairs[m * (kK / 2) + kb / 2]);
      const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
      uint32_t w[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const __half h0 = __uint2half_rn(cw[j] & 0xFFFFu), h1 = __uint2half_rn(cw[j] >> 16);
        w[j] = static_cast<uint32_t>(__half_as_ushort(h0)) | (static_cast<uint32_t>(__half_as_ushort(h1)) << 16);
      }
      *reinterpret_cast<uint4*>(a_tile + kmajor_offset(m, kb)) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    fence_proxy_async_smem();  // the tensor core reads the tile through the async proxy
    tc_fence_before();
    __syncthreads();
    // 3. counts x table into TMEM
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < kK / 16; ++kk) {
        // K = 16 per instruction = two core matrices along K
        const uint64_t adv = static_cast<uint64_t>((kk * 2 * kLBO) >> 4);
        umma_f16(tmem, a_desc0 + adv, b_desc0 + adv, idesc, kk > 0 ? 1u : 0u);
      }
      umma_commit(&mma_bar);
    }
    __syncwarp();
    if (!mbar_wait_bounded(&mma_bar, phase, kWaitLimit)) {
      if (tid == 0) {
        s_failed = 1;
        stat_add(a.stats, TBE_STAT_WAIT_TIMEOUT, 1);
      }
    }
    phase ^= 1u;
    tc_fence_after();
    // 4. readout: warp w reads TMEM lanes 32 (w % 4) .. + 31 (one bag per thread) in the 32-column
    //    chunks c0 = 32 j with j % 2 == w / 4, adds the ids past the 256th, stages the chunk in
    //    shared memory (the A tile and the count pairs are free once the MMA has completed; 16-byte
    //    slots XOR-swizzled by the row) and stores it as 128-byte row pieces, four bags per warp
    //    instruction
    {
      const int quad = warp & 3, half = warp >> 2;
      const int bag = quad * kWarp + lane;
      const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quad * kWarp) << 16);
      float4* stage = reinterpret_cast<float4*>(half == 0 ? a_tile : reinterpret_cast<uint8_t*>(pairs)) + quad * (kWarp * 8);
      int64_t ts = 0, te = 0;
      if (bag < nb) {
        te = s_off[bag + 1];
        ts = min(te, s_off[bag] + kHistIds);
      }
      for (int c0 = half * 32; c0 < a.N; c0 += 64) {
        float v[32];
        tmem_ld32(lane_addr + c0, v);  // warp-wide: every lane takes part
        if (bag < nb) {
          for (int64_t p = ts; p < te; ++p) {  // the scalar path of ids past the 256th
            const int64_t id = ld_int<IT>(a.indices, p);
            if (id < 0 || id >= a.E) continue;
            const __half* row = a.table + id * a.D + c0;
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (c0 + i < a.D) v[i] += __half2float(row[i]);
          }
        }
#pragma unroll
        for (int j = 0; j < 8; ++j)
          stage[lane * 8 + (j ^ (lane & 7))] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        __syncwarp();
#pragma unroll
        for (int it = 0; it < kWarp / 4; ++it) {
          const int r = it * 4 + (lane >> 3), j = lane & 7;  // row of the stage, 16-byte piece
          const int rb = quad * kWarp + r;                     // its bag within the tile
          if (rb < nb && c0 + 4 * j < a.D)
            __stcs(reinterpret_cast<float4*>(a.out + (b0 + rb) * a.total_D + a.col0 + c0 + 4 * j),
                   stage[r * 8 + (j ^ (r & 7))]);
        }
        __syncwarp();
      }
    }
    tc_fence_before();
    __syncthreads();  // TMEM reads done before the next tile's MMA overwrites the accumulator
    tc_fence_after();
    if (s_failed) break;
  }
  if (s_failed) {  // an MMA never signalled: wait once more (bounded) before releasing its TMEM
    mbar_wait_bounded(&mma_bar, phase ^ 1u, kWaitLimit);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------------------------------
// Backward of a counts x table feature: the table's gradient is counts^T x grad_out.
//
// "Modernizing Table Batched Embeddings with FBTriton", section 2 ("Forward-state reuse and
// preprocessing"): the backward of the small-table path can reuse the forward's per-bag counts,
// multiply them into the upstream gradient on the tensor cores with a compensated split of the
// fp32 gradient into 16-bit parts accumulating in fp32, then apply the optimizer to each row.
// The pages split into fp16 hi + lo; here each fp32 value is split exactly into three bf16
// parts (hi + mid + lo carry all 24 significand bits and keep fp32's exponent range, so no
// gradient overflows or flushes), and counts <= 256 are exact in bf16.  Per CTA and tile of 64
// bags (K = 64; two CTAs per SM):
//   1. count the first 256 ids of each bag as in the forward -- or, when the forward on the same
//      batch saved its per-bag counts ([FBT] section 2, "Forward-state reuse"), load those and
//      read no id among the first 256; ids past the 256th (rare) add their gradient row to the
//      row's fp32 sum with atomics directly;
//   2. B operand (N = E rounded up to 16, K-major): counts of row e in the tile's bags, bf16;
//      A operands (M = 128 gradient columns, K-major): the three bf16 parts of grad_out[bag, d]
//      -- a warp loads 8 bags x 32 columns coalesced and writes one 16-byte core-matrix row per
//      lane and part;
//   3. one thread issues 3 x 4 tcgen05.mma (K = 16 each) into one TMEM accumulator (128 lanes =
//      columns d, N columns = rows e) that lives across the CTA's tiles; the CTA waits on the
//      commit (bounded) before it rewrites the operands;
//   4. at the end each thread (column d) adds its accumulator row into the table's fp32 gradient
//      sum with atomics; the last CTA to finish (fence + counter) applies the optimizer once to
//      every row whose count is non-zero.
// ------------------------------------------------------------------------------------------
constexpr int kBK = 64;                        // bags per tile (the K of the MMA)
constexpr int kBM = 128;                       // gradient columns (the M of the MMA)
constexpr uint32_t kBSBO = (kBK / 8) * 128;    // 2048 B between core matrices along M/N
constexpr int kBATile = kBM * kBK * 2;         // 32 KB per bf16 split of the gradient
constexpr int kBBTile = kK * kBK * 2;          // 16 KB: counts of up to 64 rows
constexpr uint32_t kBTmemCols = 64;

struct HistBwdArgs {
  const void* indices;
  const void* offsets;
  const float* grad_out;
  __half* table;          // E x D, updated in place
  float* state;           // row-wise Adagrad state of the table's rows (NULL for SGD)
  float* gsum;            // E x D fp32 gradient sums (zeroed by the caller)
  uint32_t* rowcnt;       // E lookups per row (zeroed by the caller)
  uint32_t* done;         // CTAs finished (zeroed by the caller)
  int64_t B, num_indices, bag0;
  int E, D, N, col0, total_D;
  int opt;
  float lr, eps;
  const uint32_t* saved_pairs;  // NULL, or [B][32]: the counts the forward saved (ids not re-read)
  unsigned long long* stats;
};

__device__ __forceinline__ uint64_t smem_desc_bwd(uint32_t addr) {
  return static_cast<uint64_t>((addr >> 4) & 0x3FFF) | (static_cast<uint64_t>(kLBO >> 4) << 16) |
         (static_cast<uint64_t>(kBSBO >> 4) << 32) | (uint64_t(1) << 46);
}

// kind::f16 instruction descriptor with bf16 A and B (both K-major), fp32 accumulator.
__device__ __forceinline__ uint32_t instr_desc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ uint32_t kmajor_offset_bwd(int r, int k) {
  return static_cast<uint32_t>((r >> 3) * kBSBO + (k >> 3) * kLBO + (r & 7) * 16 + (k & 7) * 2);
}

__device__ __forceinline__ uint32_t bf16_bits(float x) {
  return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(x)));
}

// x == hi + mid + lo exactly (bf16 parts, fp32 arithmetic for the remainders).
__device__ __forceinline__ void split3(float x, uint32_t& hi, uint32_t& mid, uint32_t& lo) {
  const __nv_bfloat16 h = __float2bfloat16_rn(x);
  const float r1 = x - __bfloat162float(h);
  const __nv_bfloat16 m = __float2bfloat16_rn(r1);
  const float r2 = r1 - __bfloat162float(m);
  hi = __bfloat16_as_ushort(h);
  mid = __bfloat16_as_ushort(m);
  lo = bf16_bits(r2);
}

template <typename IT>
__global__ void __launch_bounds__(kThreads, 2) hist_bwd_kernel(HistBwdArgs a) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* a_tiles = smem;                                  // 3 x 32 KB: gradient parts
  uint8_t* b_tile = smem + 3 * kBATile;                     // 16 KB: counts
  uint32_t* pairs = reinterpret_cast<uint32_t*>(smem + 3 * kBATile + kBBTile);  // [128][32] count pairs
  __shared__ __align__(8) uint64_t mma_bar;
  __shared__ uint32_t s_tmem;
  __shared__ int s_failed, s_last;
  __shared__ int64_t s_off[kBK + 1];
  __shared__ int s_rel[kBK + 1];
  __shared__ uint32_t s_rowcnt[kK];

  const int tid = threadIdx.x, lane = lane_id(), warp = tid / kWarp;
  const bool vec_ok = (reinterpret_cast<uintptr_t>(a.indices) & 15) == 0;  // 16-byte id loads
  const int64_t tiles = (a.B + kBK - 1) / kBK;

  if (warp == 0) tmem_alloc(&s_tmem, kBTmemCols);
  if (tid == 0) {
    mbar_init(&mma_bar, 1);
    s_failed = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (tid < kK) s_rowcnt[tid] = 0;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const uint32_t idesc = instr_desc_bf16(kBM, a.N);
  const uint64_t b_desc0 = smem_desc_bwd(smem_u32(b_tile));
  uint32_t phase = 0;
  int mine = 0;  // tiles this CTA accumulated

  for (int64_t tile = blockIdx.x; tile < tiles; tile += gridDim.x, ++mine) {
    const int64_t b0 = tile * kBK;
    const int nb = static_cast<int>(min(static_cast<int64_t>(kBK), a.B - b0));
    // 1. counts of the first 256 ids of each bag: the ones the forward saved, or counted here
    if (a.saved_pairs != nullptr) {
      const uint4* src = reinterpret_cast<const uint4*>(a.saved_pairs + b0 * (kK / 2));
      for (int i = tid; i < kBK * kK / 2 / 4; i += kThreads)
        reinterpret_cast<uint4*>(pairs)[i] = i < nb * (kK / 8) ? __ldg(src + i) : make_uint4(0, 0, 0, 0);
    } else {
      for (int i = tid; i < kBK * kK / 2 / 4; i += kThreads) reinterpret_cast<uint4*>(pairs)[i] = make_uint4(0, 0, 0, 0);
    }
    for (int i = tid; i <= kBK; i += kThreads)
      s_off[i] = clamp64(ld_int<IT>(a.offsets, a.bag0 + b0 + min(i, nb)), 0, a.num_indices);
    __syncthreads();
    if (warp == 0) monotone_offsets(s_off, nb, lane);  // guard: never let a bag end before it starts
    __syncthreads();
    {
      const int64_t p0 = s_off[0];
      for (int i = tid; i <= nb; i += kThreads) s_rel[i] = static_cast<int>(s_off[i] - p0);
      __syncthreads();
      const IT* ids = static_cast<const IT*>(a.indices) + p0;
      uint32_t bad = 0;
      auto visit = [&](int r, int lo, int cur, IT id) {
        if (static_cast<uint64_t>(static_cast<int64_t>(id)) >= static_cast<uint64_t>(a.E)) {
          ++bad;
          return;
        }
        const uint32_t k = static_cast<uint32_t>(id);
        if (r - cur >= kHistIds) {
          // past the 256th id of its bag: add the bag's gradient row to row k directly
          const float4* g = reinterpret_cast<const float4*>(a.grad_out + (b0 + lo) * a.total_D + a.col0);
          float4* dst = reinterpret_cast<float4*>(a.gsum + static_cast<int64_t>(k) * a.D);
          for (int v = 0; v < a.D / 4; ++v) atomicAdd(dst + v, __ldg(g + v));
          atomicAdd(&s_rowcnt[k], 1u);
          return;
        }
        atomicAdd(&pairs[lo * (kK / 2) + (k >> 1)], (k & 1u) << 16 | (~k & 1u));
      };
      if (a.saved_pairs != nullptr) {
        // counts saved: only the ids past the 256th of each bag are read, a warp per bag
        for (int bl = warp; bl < nb; bl += kThreads / kWarp)
          for (int r = s_rel[bl] + kHistIds + lane; r < s_rel[bl + 1]; r += kWarp) visit(r, bl, s_rel[bl], __ldg(ids + r));
      } else {
        for_each_lookup<IT, kBwdVecIds, kBwdLoads, kThreads / kWarp>(ids, p0, vec_ok, s_rel, nb, warp, lane, visit);
      }
      if (bad) stat_add(a.stats, TBE_STAT_UNREPAIRED, bad);
    }
    __syncthreads();
    // row totals of the tile
    if (tid < a.E) {
      uint32_t tot = 0;
      for (int k = 0; k < nb; ++k) tot += (pairs[k * (kK / 2) + (tid >> 1)] >> ((tid & 1) * 16)) & 0xFFFFu;
      s_rowcnt[tid] += tot;
    }
    // 2a. B operand: element (row e, bag k) = count, 8 bags per 16-byte core-matrix row
    for (int q = tid; q < a.N * (kBK / 8); q += kThreads) {
      const int e = q / (kBK / 8), kb = (q % (kBK / 8)) * 8;
      uint32_t w[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t c0 = (pairs[(kb + 2 * j) * (kK / 2) + (e >> 1)] >> ((e & 1) * 16)) & 0xFFFFu;
        const uint32_t c1 = (pairs[(kb + 2 * j + 1) * (kK / 2) + (e >> 1)] >> ((e & 1) * 16)) & 0xFFFFu;
        w[j] = bf16_bits(static_cast<float>(c0)) | (bf16_bits(static_cast<float>(c1)) << 16);
      }
      *reinterpret_cast<uint4*>(b_tile + kmajor_offset_bwd(e, kb)) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    // 2b. A operands: element (column d, bag k) of each bf16 part of the gradient
    //     A warp loads the gradient values of all its core-matrix rows (four per warp: 32 per
    //     lane in flight) before splitting and writing any of them.
    {
      constexpr int NT = (kBM / kWarp) * (kBK / 8);  // 16-byte core-matrix rows per part
      constexpr int NW = kThreads / kWarp;
      constexpr int TPASS = (NT + NW - 1) / NW;
      for (int t0 = warp; t0 < NT; t0 += TPASS * NW) {
        float g[TPASS][8];
#pragma unroll
        for (int p = 0; p < TPASS; ++p) {
          const int task = t0 + p * NW;
          const int d = (task % (kBM / kWarp)) * kWarp + lane;
          const int kb = (task / (kBM / kWarp)) * 8;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int k = kb + j;
            g[p][j] = (task < NT && d < a.D && k < nb) ? __ldg(a.grad_out + (b0 + k) * a.total_D + a.col0 + d) : 0.f;
          }
        }
#pragma unroll
        for (int p = 0; p < TPASS; ++p) {
          const int task = t0 + p * NW;
          if (task >= NT) break;
          const int d = (task % (kBM / kWarp)) * kWarp + lane;
          const int kb = (task / (kBM / kWarp)) * 8;
          uint32_t hw[4], mw[4], lw[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            uint32_t h0, m0, l0, h1, m1, l1;
            split3(g[p][2 * j], h0, m0, l0);
            split3(g[p][2 * j + 1], h1, m1, l1);
            hw[j] = h0 | (h1 << 16);
            mw[j] = m0 | (m1 << 16);
            lw[j] = l0 | (l1 << 16);
          }
          const uint32_t off = kmajor_offset_bwd(d, kb);
          *reinterpret_cast<uint4*>(a_tiles + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          *reinterpret_cast<uint4*>(a_tiles + kBATile + off) = make_uint4(mw[0], mw[1], mw[2], mw[3]);
          *reinterpret_cast<uint4*>(a_tiles + 2 * kBATile + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    // 3. gradient parts x counts into the accumulator
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int part = 0; part < 3; ++part) {
        const uint64_t a_desc0 = smem_desc_bwd(smem_u32(a_tiles + part * kBATile));
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk) {
          const uint64_t adv = static_cast<uint64_t>((kk * 2 * kLBO) >> 4);
          umma_f16(tmem, a_desc0 + adv, b_desc0 + adv, idesc, (mine > 0 || part > 0 || kk > 0) ? 1u : 0u);
        }
      }
      umma_commit(&mma_bar);
    }
    __syncwarp();
    if (!mbar_wait_bounded(&mma_bar, phase, kWaitLimit)) {
      if (tid == 0) {
        s_failed = 1;
        stat_add(a.stats, TBE_STAT_WAIT_TIMEOUT, 1);
      }
    }
    phase ^= 1u;
    tc_fence_after();
    __syncthreads();  // operands free for the next tile; s_failed visible
    if (s_failed) break;
  }
  if (s_failed) mbar_wait_bounded(&mma_bar, phase ^ 1u, kWaitLimit);

  // 4. this CTA's sums into the table's: thread = column d (warps 0-3), accumulator column = row e
  if (mine > 0 && !s_failed && warp < kBM / kWarp) {
    const int d = tid;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(warp * kWarp) << 16);
    for (int c0 = 0; c0 < a.N; c0 += 32) {
      float v[32];
      tmem_ld32(lane_addr + c0, v);
      if (d < a.D) {
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (c0 + i < a.E) atomicAdd(a.gsum + static_cast<int64_t>(c0 + i) * a.D + d, v[i]);
      }
    }
  }
  if (tid < a.E && s_rowcnt[tid] > 0) atomicAdd(a.rowcnt + tid, s_rowcnt[tid]);
  __threadfence();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kBTmemCols);
  if (tid == 0) s_last = atomicAdd(a.done, 1u) == gridDim.x - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();  // acquire: every CTA's sums, published before its increment
  // the optimizer, once per touched row: warp per row, lane over float4 slices
  for (int e = warp; e < a.E; e += kThreads / kWarp) {
    if (__ldcg(a.rowcnt + e) == 0) continue;  // untouched rows are not written
    const int nv = a.D / 4;
    float g[4][4];
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int v = lane + j * kWarp;
      float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
      if (v < nv) f = __ldcg(reinterpret_cast<const float4*>(a.gsum + static_cast<int64_t>(e) * a.D) + v);
      g[j][0] = f.x;
      g[j][1] = f.y;
      g[j][2] = f.z;
      g[j][3] = f.w;
      ss += f.x * f.x + f.y * f.y + f.z * f.z + f.w * f.w;
    }
    float scale = a.lr;
    if (a.opt == TBE_OPT_ROWWISE_ADAGRAD) {
      for (int m = 16; m > 0; m >>= 1) ss += __shfl_xor_sync(FULL, ss, m);
      const float s_new = a.state[e] + ss / static_cast<float>(a.D);
      __syncwarp();
      if (lane == 0) a.state[e] = s_new;
      scale = a.lr / (sqrtf(s_new) + a.eps);
    }
    __half* row = a.table + static_cast<int64_t>(e) * a.D;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int v = lane + j * kWarp;
      if (v < nv) {
        uint2 raw = reinterpret_cast<const uint2*>(row)[v];
        __half2 p0 = *reinterpret_cast<__half2*>(&raw.x), p1 = *reinterpret_cast<__half2*>(&raw.y);
        const float2 f0 = __half22float2(p0), f1 = __half22float2(p1);
        p0 = __floats2half2_rn(f0.x - scale * g[j][0], f0.y - scale * g[j][1]);
        p1 = __floats2half2_rn(f1.x - scale * g[j][2], f1.y - scale * g[j][3]);
        raw.x = *reinterpret_cast<uint32_t*>(&p0);
        raw.y = *reinterpret_cast<uint32_t*>(&p1);
        reinterpret_cast<uint2*>(row)[v] = raw;
      }
    }
  }
}

}  // namespace

bool histogram_supported() { return true; }

cudaError_t launch_forward_histogram(const Problem& P, const tbe_tables& tab, const void* weights,
                                     const void* indices, const void* offsets, float* out, int table,
                                     bool fused_bounds, uint32_t* save_pairs, unsigned long long* stats,
                                     const DeviceInfo& dev, cudaStream_t s) {
  (void)tab;
  int64_t woff = 0, col0 = 0;
  for (int t = 0; t < table; ++t) {
    woff += P.E[t] * P.D[t];
    col0 += P.D[t];
  }
  HistArgs a;
  a.table = static_cast<const __half*>(weights) + woff;
  a.indices = indices;
  a.offsets = offsets;
  a.out = out;
  a.B = P.B;
  a.num_indices = P.num_indices;
  a.bag0 = static_cast<int64_t>(table) * P.B;
  a.E = static_cast<int>(P.E[table]);
  a.D = P.D[table];
  a.N = (a.D + 15) / 16 * 16;
  a.col0 = static_cast<int>(col0);
  a.total_D = P.total_D;
  a.fused_bounds = fused_bounds ? 1 : 0;
  a.save_pairs = save_pairs;
  a.stats = stats;
  if (P.B == 0) return cudaSuccess;
  const size_t smem = 3 * kTileBytes + 1024;  // A, B, count pairs + alignment slack
  auto k = P.itype == TBE_I32 ? hist_tc_kernel<int32_t> : hist_tc_kernel<int64_t>;
  // opt-in shared memory is a per-device function attribute: set it once per device
  static std::atomic<uint64_t> attr_set[2] = {{0}, {0}};
  int dev_id = 0;
  cudaError_t e = cudaGetDevice(&dev_id);
  if (e != cudaSuccess) return e;
  const uint64_t bit = uint64_t(1) << (dev_id & 63);
  std::atomic<uint64_t>& flag = attr_set[P.itype == TBE_I32 ? 0 : 1];
  if ((flag.load() & bit) == 0) {
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    flag.fetch_or(bit);
  }
  const int64_t tiles = (P.B + kM - 1) / kM;
  // at most 4 CTAs per SM: 4 x 128 TMEM columns fit in the SM's 512 without waiting
  int64_t grid = static_cast<int64_t>(dev.sms) * 4;
  if (tiles < grid) grid = tiles;
  k<<<static_cast<int>(grid), kThreads, smem, s>>>(a);
  note_launch();
  return cudaGetLastError();
}

size_t hist_backward_ws_bytes() { return kHistWsBytes; }

cudaError_t launch_backward_histogram(const Problem& P, const BwdCtx& c, int table, void* hist_ws,
                                      const uint32_t* saved_pairs, tbe_optimizer opt, const DeviceInfo& dev,
                                      cudaStream_t s) {
  int64_t woff = 0, roff = 0, col0 = 0;
  for (int t = 0; t < table; ++t) {
    woff += P.E[t] * P.D[t];
    roff += P.E[t];
    col0 += P.D[t];
  }
  HistBwdArgs a;
  a.indices = c.indices;
  a.offsets = c.offsets;
  a.grad_out = c.grad_out;
  a.table = static_cast<__half*>(c.weights) + woff;
  a.state = c.state == nullptr ? nullptr : c.state + roff;
  char* ws = static_cast<char*>(hist_ws);
  a.gsum = reinterpret_cast<float*>(ws);
  a.rowcnt = reinterpret_cast<uint32_t*>(ws + kHistGsumBytes);
  a.done = a.rowcnt + kK;
  a.B = P.B;
  a.num_indices = P.num_indices;
  a.bag0 = static_cast<int64_t>(table) * P.B;
  a.E = static_cast<int>(P.E[table]);
  a.D = P.D[table];
  a.N = (a.E + 15) / 16 * 16;
  a.col0 = static_cast<int>(col0);
  a.total_D = P.total_D;
  a.opt = opt;
  a.lr = c.lr;
  a.eps = c.eps;
  a.saved_pairs = saved_pairs;
  a.stats = c.stats;
  if (P.B == 0) return cudaSuccess;
  const size_t smem = 3 * kBATile + kBBTile + kBK * kK * 2 + 1024;
  auto k = P.itype == TBE_I32 ? hist_bwd_kernel<int32_t> : hist_bwd_kernel<int64_t>;
  static std::atomic<uint64_t> attr_set[2] = {{0}, {0}};
  int dev_id = 0;
  cudaError_t e = cudaGetDevice(&dev_id);
  if (e != cudaSuccess) return e;
  const uint64_t bit = uint64_t(1) << (dev_id & 63);
  std::atomic<uint64_t>& flag = attr_set[P.itype == TBE_I32 ? 0 : 1];
  if ((flag.load() & bit) == 0) {
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    flag.fetch_or(bit);
  }
  const int64_t tiles = (P.B + kBK - 1) / kBK;
  int64_t grid = 2 * static_cast<int64_t>(dev.sms);  // two CTAs per SM (65 KB of shared memory each)
  if (tiles < grid) grid = tiles;
  k<<<static_cast<int>(grid), kThreads, smem, s>>>(a);
  note_launch();
  return cudaGetLastError();
}

}  // namespace tbe
