// tbe_internal.cuh -- internal types, device helpers and launcher declarations shared by the
// translation units of the TBE library.  Nothing here is part of the C interface (tbe.h).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <type_traits>
#include <vector>

#include "tbe.h"

namespace tbe {

constexpr int kWarp = 32;
constexpr int kMaxTables = 4096;
constexpr int kNumBuckets = TBE_NUM_BUCKETS;  // short-run buckets: next_pow2(D) = 2^k
constexpr int kMaxD = 1024;
// Most lookups a problem may hold.  Kernels keep lookup positions in 32-bit ints and compute
// positions up to 127 past a bag's end (the gather's 32-position id windows run up to four
// windows ahead); 2^16 below 2^31 keeps every such position representable.
constexpr int64_t kMaxIndices = (int64_t(1) << 31) - (int64_t(1) << 16);
constexpr int kSortThreads = 256;
constexpr int kSortItems = 16;
constexpr int kSortTile = kSortThreads * kSortItems;  // keys per radix-sort tile
constexpr int kMaxRadixBits = 10;                     // digits of 8..10 bits: passes = ceil(bits/10)
constexpr int kMaxRadixPasses = 4;                    // 32-bit keys
constexpr int kMaxRadix = 1 << kMaxRadixBits;
constexpr int kExpandBags = 512;                        // bags per expand CTA

// ------------------------------------------------------------------------------------------
// Host-side validated problem and device description
// ------------------------------------------------------------------------------------------
struct Problem {
  int T = 0;
  int64_t B = 0, TB = 0, num_indices = 0;
  int wdtype = 0, itype = 0;
  bool weighted = false;
  int pooling = 0;          // tbe_pooling
  bool scaled = false;      // the backward's sort carries a per-lookup factor (psw, over L for mean pooling)
  bool mean_inv = false;    // unweighted mean pooling: the update kernels scale by 1 / L of the bag
  std::vector<int> D;
  std::vector<int64_t> E;
  std::vector<uint8_t> long_bags;
  int64_t total_rows = 0;
  int total_D = 0, max_D = 0;
  int wbytes = 0;           // bytes per weight element
  int vec_bytes = 16;       // width of one weight-row load (16 or 8 bytes)
};

struct DeviceInfo {
  int id = 0;
  int sms = 0;
};

// Tables whose backward goes through counts^T x grad_out on the tensor cores (the forward's
// counts x table tables): at most kMaxHistTables per call, each with kHistWsBytes of workspace
// zeroed per call (fp32 gradient sums of up to 64 x 128, row counts, a CTA counter).  Their
// lookups stay out of the sort.
constexpr int kMaxHistTables = 8;
constexpr size_t kHistGsumBytes = 64 * 128 * 4;
constexpr size_t kHistWsBytes = kHistGsumBytes + 512;
bool hist_forward_eligible(const Problem& P, const tbe_options& o, int t);

tbe_status make_problem(const tbe_problem* p, Problem* out);

// TBE_OK for cudaSuccess; otherwise records e as this thread's last CUDA error (reported by
// tbe_last_cuda_error) and returns TBE_ERR_CUDA.
tbe_status cuda_status(cudaError_t e);

// Counts kernel launches of the current call on this host thread (reported through
// tbe_options.launch_counter).
void note_launch(int n = 1);
tbe_status device_info(DeviceInfo* out);

// Layout of the backward workspace (byte offsets from the 256-aligned base).
struct BwdLayout {
  size_t counters = 0, keys[2] = {0, 0}, vals[2] = {0, 0}, psw[2] = {0, 0};
  size_t sort_counts = 0, sort_totals = 0, rle_counts = 0, unique = 0, run_off = 0, run_len = 0;
  size_t short_list[kNumBuckets] = {0};
  size_t long_list = 0, chunks = 0, countdown = 0, ws_rows = 0, cls_counts = 0;
  size_t inv_len = 0;  // unweighted mean pooling: 1 / L per bag (TB floats)
  size_t total = 0;
  uint32_t short_cap[kNumBuckets] = {0};
  uint32_t long_cap = 0, chunk_cap = 0, u_cap = 0, n_cap = 0;
  int sort_grid = 1, rle_grid = 1, cls_grid = 1, key_bits = 1, passes = 1, radix_bits = 8, final_buf = 0;
  int pass_bits[4] = {8, 8, 8, 8};  // digit width of each radix pass, low digit first; radix_bits = the widest
  int acc_bytes = 4;  // fp32 workspace rows (fp64 for fp32 tables)
  size_t hist_ws = 0;  // nhist x kHistWsBytes
  int nhist = 0;
  int hist_t[kMaxHistTables] = {0};
};

BwdLayout make_bwd_layout(const Problem& P, const tbe_options& opt, const DeviceInfo& dev);

// Grid size of a persistent launch: resident blocks per SM (occupancy) x SMs, at most `cap`.
template <typename K>
int persistent_grid(K kernel, int threads, size_t smem, const DeviceInfo& dev, int64_t cap) {
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  int64_t g = static_cast<int64_t>(per_sm) * dev.sms;
  if (cap < g) g = cap;
  return g < 1 ? 1 : static_cast<int>(g);
}

// ------------------------------------------------------------------------------------------
// Device pointers for the backward pipeline
// ------------------------------------------------------------------------------------------
struct BwdCtx {
  // problem
  int T;
  int64_t B, TB, num_indices, total_rows;
  int total_D, max_D;
  int threshold, chunk;
  // tables
  const int64_t* woff;
  const int32_t* doff;
  const int64_t* roff;
  // inputs / state
  void* weights;
  float* state;
  const void* indices;
  const void* offsets;
  const float* psw;
  const float* grad_out;
  float lr, eps;
  float* inv_len;                   // [TB] 1 / L of each bag (unweighted mean pooling), else NULL
  // workspace
  uint32_t* counters;
  uint32_t* keys[2];
  uint32_t* vals[2];
  float* pswbuf[2];
  uint32_t* sort_counts;
  uint32_t* sort_totals;
  uint32_t* rle_counts;
  uint32_t* unique;
  uint32_t* run_off;
  uint32_t* run_len;
  uint4* short_list[kNumBuckets];  // per short run: {first lookup, length, key, table}
  uint32_t short_cap[kNumBuckets];
  uint32_t* long_list;              // run id of each long run (its slot)
  uint4* chunks;                    // per chunk: {first lookup, end, key, slot}
  uint32_t* countdown;
  void* ws_rows;
  uint32_t long_cap, chunk_cap, u_cap;
  int sort_grid, rle_grid, cls_grid;
  uint32_t* cls_counts;             // [lists][cls_grid] per-block counts, then their prefixes
  unsigned long long* stats;
  int nhist;                        // tables on the counts path (their lookups skip the sort)
  int hist_t[kMaxHistTables];
  char* hist_ws;
};

// ------------------------------------------------------------------------------------------
// Launchers (one translation unit each group); all asynchronous on `s`
// ------------------------------------------------------------------------------------------
cudaError_t launch_bounds(const Problem& P, const tbe_tables& tab, void* indices, void* offsets,
                          int64_t* ws, int grid, unsigned long long* stats, bool with_ids, cudaStream_t s);
int bounds_grid(const DeviceInfo& dev);

cudaError_t launch_forward_gather(const Problem& P, const tbe_tables& tab, const void* weights,
                                  void* indices, const void* offsets, const float* psw, float* out,
                                  int64_t unit_begin, int64_t unit_end, bool fused_bounds, bool allow_tma,
                                  unsigned long long* stats, const DeviceInfo& dev, cudaStream_t s);

cudaError_t launch_forward_long_bags(const Problem& P, const tbe_tables& tab, const void* weights,
                                     const void* indices, const void* offsets, const float* psw, float* out,
                                     int64_t unit_begin, int64_t unit_end, const DeviceInfo& dev, cudaStream_t s);

bool histogram_supported();
// saved_pairs / save_pairs: NULL, or the table's per-bag counts ([B][32] words, two 16-bit
// counts each) that the forward saves and a backward on the same batch reads instead of the ids
cudaError_t launch_backward_histogram(const Problem& P, const BwdCtx& c, int table, void* hist_ws,
                                      const uint32_t* saved_pairs, tbe_optimizer opt, const DeviceInfo& dev,
                                      cudaStream_t s);
cudaError_t launch_forward_histogram(const Problem& P, const tbe_tables& tab, const void* weights,
                                     const void* indices, const void* offsets, float* out, int table,
                                     bool fused_bounds, uint32_t* save_pairs, unsigned long long* stats,
                                     const DeviceInfo& dev, cudaStream_t s);
// Bytes of the per-bag counts of one counts x table table, saved by the forward.
constexpr size_t kHistPairsBytesPerBag = 32 * sizeof(uint32_t);

cudaError_t launch_psw_gradient(const Problem& P, const tbe_tables& tab, const void* weights,
                                const void* indices, const void* offsets, const float* grad_out,
                                float* grad_psw, const DeviceInfo& dev, cudaStream_t s);

cudaError_t launch_expand(const Problem& P, const BwdCtx& c, cudaStream_t s);
cudaError_t launch_sort(const Problem& P, const BwdCtx& c, const BwdLayout& L, cudaStream_t s);
cudaError_t launch_rle(const Problem& P, const BwdCtx& c, const BwdLayout& L, cudaStream_t s);
cudaError_t launch_classify(const Problem& P, const BwdCtx& c, const DeviceInfo& dev, int mode, cudaStream_t s);
cudaError_t launch_short_updates(const Problem& P, const BwdCtx& c, const BwdLayout& L,
                                 tbe_optimizer opt, int scheduler, const DeviceInfo& dev,
                                 cudaStream_t s);
cudaError_t launch_long_updates(const Problem& P, const BwdCtx& c, const BwdLayout& L,
                                tbe_optimizer opt, bool fused, int scheduler, int merge,
                                const DeviceInfo& dev, cudaStream_t s);
cudaError_t launch_long_apply(const Problem& P, const BwdCtx& c, const BwdLayout& L,
                              tbe_optimizer opt, const DeviceInfo& dev, cudaStream_t s);

// ------------------------------------------------------------------------------------------
// Device helpers
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ int lane_id() { return threadIdx.x & (kWarp - 1); }

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

template <typename IT>
__device__ __forceinline__ int64_t ld_int(const void* p, int64_t i) {
  return static_cast<int64_t>(__ldg(static_cast<const IT*>(p) + i));
}

__device__ __forceinline__ int64_t clamp64(int64_t v, int64_t lo, int64_t hi) {
  return v < lo ? lo : (v > hi ? hi : v);
}

__device__ __forceinline__ void stat_add(unsigned long long* stats, int k, unsigned long long v) {
  if (stats != nullptr && v != 0) atomicAdd(stats + k, v);
}

// Debug build (-DTBE_CHECKED=1): device-side range checks on indices the kernels derive from
// data (sorted positions, run bounds, list slots), each failure counted in
// stats[TBE_STAT_CHECK_FAILED] and the access skipped -- an error counter, never a trap.
//   TBE_CHECK(ok, stats)  a check only the debug build has (true, not evaluated, otherwise)
//   TBE_GUARD(ok, stats)  a guard every build keeps; the debug build also counts its failures
#ifndef TBE_CHECKED
#define TBE_CHECKED 0
#endif
__device__ __forceinline__ bool check_count(bool ok, unsigned long long* stats) {
#if TBE_CHECKED
  if (!ok) stat_add(stats, TBE_STAT_CHECK_FAILED, 1);
#endif
  return ok;
}
#define TBE_CHECK(ok, stats) (!TBE_CHECKED || ::tbe::check_count((ok), (stats)))
#define TBE_GUARD(ok, stats) (::tbe::check_count((ok), (stats)))

// Table of a linear row id: the t with row_offsets[t] <= key < row_offsets[t+1].
__device__ __forceinline__ int table_of_row(const int64_t* roff, int T, int64_t key) {
  int lo = 0, hi = T;  // invariant: roff[lo] <= key < roff[hi]
  while (hi - lo > 1) {
    int mid = (lo + hi) >> 1;
    if (__ldg(roff + mid) <= key) lo = mid;
    else hi = mid;
  }
  return lo;
}

// Weight element traits: accumulation type (fp32 for 16-bit tables, fp64 for fp32 tables,
// as the forward's accumulation rule states) and vector conversions.
template <typename WT> struct WTraits;
template <> struct WTraits<float> {
  using Acc = double;
};
template <> struct WTraits<__half> {
  using Acc = float;
};
template <> struct WTraits<__nv_bfloat16> {
  using Acc = float;
};

template <int BYTES> struct RawVec;
template <> struct RawVec<16> { using T = uint4; };
template <> struct RawVec<8> { using T = uint2; };
template <> struct RawVec<4> { using T = uint32_t; };

__device__ __forceinline__ void raw_words(const uint4& v, uint32_t (&w)[4]) { w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w; }
__device__ __forceinline__ void raw_words(const uint2& v, uint32_t (&w)[2]) { w[0] = v.x; w[1] = v.y; }
__device__ __forceinline__ void raw_words(const uint32_t& v, uint32_t (&w)[1]) { w[0] = v; }
__device__ __forceinline__ uint4 make_raw(const uint32_t (&w)[4]) { return make_uint4(w[0], w[1], w[2], w[3]); }
__device__ __forceinline__ uint2 make_raw(const uint32_t (&w)[2]) { return make_uint2(w[0], w[1]); }
__device__ __forceinline__ uint32_t make_raw(const uint32_t (&w)[1]) { return w[0]; }

// Unpack a raw vector of weights into N accumulator values.
template <typename WT, int BYTES>
struct VecIO {
  static constexpr int N = BYTES / static_cast<int>(sizeof(WT));
  static constexpr int W = BYTES / 4;
  using Raw = typename RawVec<BYTES>::T;
  using Acc = typename WTraits<WT>::Acc;

  __device__ __forceinline__ static void unpack(const Raw& r, float (&f)[N]) {
    uint32_t w[W];
    raw_words(r, w);
#pragma unroll
    for (int i = 0; i < W; ++i) {
      if constexpr (sizeof(WT) == 2) {
        float2 p;
        if constexpr (std::is_same<WT, __half>::value) {
          __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
          p = __half22float2(h);
        } else {
          __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(&w[i]);
          p = __bfloat1622float2(h);
        }
        f[2 * i] = p.x;
        f[2 * i + 1] = p.y;
      } else {
        f[i] = __uint_as_float(w[i]);
      }
    }
  }

  // Round-to-nearest-even store of N values.
  __device__ __forceinline__ static Raw pack(const float (&f)[N]) {
    uint32_t w[W];
#pragma unroll
    for (int i = 0; i < W; ++i) {
      if constexpr (sizeof(WT) == 2) {
        if constexpr (std::is_same<WT, __half>::value) {
          __half2 h = __floats2half2_rn(f[2 * i], f[2 * i + 1]);
          w[i] = *reinterpret_cast<uint32_t*>(&h);
        } else {
          __nv_bfloat162 h = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
          w[i] = *reinterpret_cast<uint32_t*>(&h);
        }
      } else {
        w[i] = __float_as_uint(f[i]);
      }
    }
    return make_raw(w);
  }
};

// ------------------------------------------------------------------------------------------
// Shared-memory staging with bulk copies (sm_90+ PTX): one lane copies one whole row into
// shared memory; completion is counted in bytes on an mbarrier.
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Arrive once on the barrier and add `bytes` to the bytes it waits for.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n"
      "  .reg .pred p;\n"
      "  mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      "  selp.u32 %0, 1, 0, p;\n"
      "}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase of the given parity; gives up after `limit` polls (each poll suspends
// for a hardware-chosen time) and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint32_t limit) {
  for (uint32_t i = 0; i < limit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}

// Bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned) global -> shared,
// completion counted in bytes on the mbarrier.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Orders this thread's earlier shared-memory accesses before later bulk-copy (async proxy)
// accesses of the same memory, and makes barrier initialisation visible to it.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Bulk reduction (sm_90+): global[dst .. dst+bytes) += shared[src ..), element type Acc (f32 or
// f64), performed by the async proxy in L2.  bytes is a multiple of 16, both addresses 16-byte
// aligned.  Waits until the additions have been performed, then orders them before this
// thread's later generic-proxy accesses of global memory.
template <typename Acc>
__device__ __forceinline__ void bulk_reduce_add(void* dst, const void* src, uint32_t bytes) {
  if constexpr (sizeof(Acc) == 8) {
    asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f64 [%0], [%1], %2;" ::"l"(dst),
                 "r"(smem_u32(src)), "r"(bytes)
                 : "memory");
  } else {
    asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;" ::"l"(dst),
                 "r"(smem_u32(src)), "r"(bytes)
                 : "memory");
  }
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Cluster launch control (sm_100+).  clc_init by one thread before a __syncthreads; clc_steal
// by every thread of the CTA: it asks the hardware to cancel a CTA of this grid that has not
// started, and returns that CTA's x index (whose work the caller then does) or -1 when none is
// left.  The response wait is bounded; on time-out the CTA counts TBE_STAT_WAIT_TIMEOUT, waits
// once more for the response (bounded) and stops stealing.
constexpr uint32_t kClcWaitLimit = 1u << 22;

__device__ __forceinline__ void clc_init(uint64_t* bar) {
  mbar_init(bar, 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ int64_t clc_steal(uint4* resp, uint64_t* bar, int64_t* next, uint32_t& phase,
                                             unsigned long long* stats) {
  __syncthreads();  // every warp is done with the current block (and has read *next)
  if (threadIdx.x == 0) {
    int64_t nb = -1;
    mbar_arrive_expect_tx(bar, 16);
    asm volatile("clusterlaunchcontrol.try_cancel.async.shared::cta.mbarrier::complete_tx::bytes.b128 [%0], [%1];" ::"r"(
                     smem_u32(resp)),
                 "r"(smem_u32(bar))
                 : "memory");
    if (mbar_wait_bounded(bar, phase, kClcWaitLimit)) {
      uint32_t cancelled = 0, x = 0;
      asm volatile(
          "{\n\t.reg .b128 r;\n\t.reg .pred p;\n\tld.shared.b128 r, [%2];\n\t"
          "clusterlaunchcontrol.query_cancel.is_canceled.pred.b128 p, r;\n\tselp.u32 %0, 1, 0, p;\n\t"
          "clusterlaunchcontrol.query_cancel.get_first_ctaid::x.b32.b128 %1, r;\n\t}"
          : "=r"(cancelled), "=r"(x)
          : "r"(smem_u32(resp))
          : "memory");
      if (cancelled) nb = x;
    } else {
      stat_add(stats, TBE_STAT_WAIT_TIMEOUT, 1);
      mbar_wait_bounded(bar, phase, kClcWaitLimit);
    }
    *next = nb;
  }
  phase ^= 1u;
  __syncthreads();
  return *next;
}

template <typename Raw>
__device__ __forceinline__ Raw ldg_raw(const Raw* p) {
  return __ldg(p);
}
template <>
__device__ __forceinline__ uint32_t ldg_raw<uint32_t>(const uint32_t* p) {
  return __ldg(p);
}

}  // namespace tbe
