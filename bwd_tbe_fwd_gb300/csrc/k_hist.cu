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
// accumulator and keeps the table in shared memory as the B operand.  Per tile of 128 bags:
//   1. the tile's 129 offsets go to shared memory; all 256 threads stream the tile's contiguous
//      id range with 16 coalesced loads in flight each, find every id's bag by binary search over
//      the offsets, and for ids among the first 256 of their bag count them with 32-bit
//      shared-memory atomics on packed 16-bit pairs; the counts are then written as the fp16 A
//      tile (counts <= 256 are exact in fp16) in the canonical K-major layout without swizzle
//      (8 x 16-byte core matrices);
//   2. one thread issues four tcgen05.mma.cta_group::1.kind::f16 (M=128, N=D rounded up to 16,
//      K=16 each) and commits them to an mbarrier; the CTA waits on it (bounded);
//   3. warps 0-3 read their 32 accumulator lanes each (one bag per thread) with tcgen05.ld
//      32x32b.x32, add the rows of ids past the 256th, and store the pooled row.
// Counts x table is exact up to fp32 rounding, so the result equals the gather's sum.
#include <atomic>

#include "tbe_internal.cuh"

namespace tbe {
namespace {

constexpr int kThreads = 256;       // 8 warps count; warps 0-3 (one bag per thread) read TMEM
constexpr int kIdsPerThread = 16;   // ids in flight per thread while counting
constexpr int kM = 128;
constexpr int kK = 64;              // E padded to 64
constexpr int kMaxN = 128;          // D <= 128
constexpr int kHistIds = 256;       // ids per bag counted by the histogram
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
  const int64_t tiles = (a.B + kM - 1) / kM;

  // TMEM for the accumulator (warp 0 allocates for the CTA), the MMA completion barrier
  if (warp == 0) tmem_alloc(&s_tmem, kTmemCols);
  if (tid == 0) {
    mbar_init(&mma_bar, 1);
    s_failed = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // B tile: element (n, k) = W[k][n] for k < E and n < D, zero elsewhere
  for (int q = tid; q < kMaxN * (kK / 8); q += kThreads) {
    const int n = q / (kK / 8), kb = (q % (kK / 8)) * 8;
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int k0 = kb + 2 * j, k1 = k0 + 1;
      const __half h0 = (k0 < a.E && n < a.D) ? a.table[static_cast<int64_t>(k0) * a.D + n] : __float2half(0.f);
      const __half h1 = (k1 < a.E && n < a.D) ? a.table[static_cast<int64_t>(k1) * a.D + n] : __float2half(0.f);
      w[j] = static_cast<uint32_t>(__half_as_ushort(h0)) | (static_cast<uint32_t>(__half_as_ushort(h1)) << 16);
    }
    *reinterpret_cast<uint4*>(b_tile + kmajor_offset(n, kb)) = make_uint4(w[0], w[1], w[2], w[3]);
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const uint32_t idesc = instr_desc(kM, a.N);
  const uint64_t a_desc0 = smem_desc(smem_u32(a_tile)), b_desc0 = smem_desc(smem_u32(b_tile));
  uint32_t phase = 0;

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
    for (int i = 1; i <= nb; ++i) {  // guard: never let a bag end before it starts
      if (tid == 0 && s_off[i] < s_off[i - 1]) s_off[i] = s_off[i - 1];
    }
    __syncthreads();
    {
      // positions relative to the tile's first lookup (32-bit), bag starts in shared memory
      const int64_t p0 = s_off[0];
      const int rel_end = static_cast<int>(s_off[nb] - p0);
      for (int i = tid; i <= nb; i += kThreads) s_rel[i] = static_cast<int>(s_off[i] - p0);
      __syncthreads();
      const IT* ids = static_cast<const IT*>(a.indices) + p0;
      uint32_t bad = 0;
      int lo = 0, cur = 0, nxt = nb > 0 ? s_rel[1] : 0x7fffffff;  // this thread's bag and its bounds
      for (int base = 0; base < rel_end; base += kThreads * kIdsPerThread) {
        IT id[kIdsPerThread];
#pragma unroll
        for (int j = 0; j < kIdsPerThread; ++j) {
          const int r = base + j * kThreads + tid;
          id[j] = r < rel_end ? __ldg(ids + r) : IT(0);
        }
#pragma unroll
        for (int j = 0; j < kIdsPerThread; ++j) {
          const int r = base + j * kThreads + tid;
          if (r >= rel_end) continue;
          while (r >= nxt) {  // positions only increase: walk forward to r's bag
            ++lo;
            cur = nxt;
            nxt = lo + 1 <= nb ? s_rel[lo + 1] : 0x7fffffff;
          }
          if (r - cur >= kHistIds) continue;  // the scalar path adds it
          if (static_cast<uint64_t>(static_cast<int64_t>(id[j])) >= static_cast<uint64_t>(a.E)) {
            ++bad;
            continue;
          }
          const uint32_t k = static_cast<uint32_t>(id[j]);
          // two 16-bit counts per word (counts <= 256 never carry into the neighbour)
          atomicAdd(&pairs[lo * (kK / 2) + (k >> 1)], (k & 1u) << 16 | (~k & 1u));
        }
      }
      if (bad) stat_add(a.stats, TBE_STAT_UNREPAIRED, bad);
    }
    __syncthreads();
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
    // 3. warps 0-3 read their bag rows out of TMEM, add the ids past the 256th, store
    if (warp < kM / kWarp) {
      const int64_t b = b0 + tid;
      const uint32_t lane_addr = tmem + (static_cast<uint32_t>(warp * kWarp) << 16);
      int64_t ts = 0, te = 0;
      if (tid < nb) {
        te = s_off[tid + 1];
        ts = min(te, s_off[tid] + kHistIds);
      }
      for (int c0 = 0; c0 < a.N; c0 += 32) {
        float v[32];
        tmem_ld32(lane_addr + c0, v);  // warp-wide: every lane takes part
        if (tid < nb) {
          for (int64_t p = ts; p < te; ++p) {  // the scalar path of ids past the 256th
            const int64_t id = ld_int<IT>(a.indices, p);
            if (id < 0 || id >= a.E) continue;
            const __half* row = a.table + id * a.D + c0;
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (c0 + i < a.D) v[i] += __half2float(row[i]);
          }
          float* orow = a.out + b * a.total_D + a.col0 + c0;
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            if (c0 + i < a.D) __stcs(reinterpret_cast<float4*>(orow + i), make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]));
        }
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

}  // namespace

bool histogram_supported() { return true; }

cudaError_t launch_forward_histogram(const Problem& P, const tbe_tables& tab, const void* weights,
                                     const void* indices, const void* offsets, float* out, int table,
                                     unsigned long long* stats, const DeviceInfo& dev, cudaStream_t s) {
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

}  // namespace tbe
