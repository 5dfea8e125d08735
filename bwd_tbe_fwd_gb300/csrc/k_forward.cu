// k_forward.cu -- pooled forward gather.
//
// "Modernizing Table Batched Embeddings with FBTriton", section 2 ("The general gather
// path"): for each table and bag, gather the indexed rows, optionally scale them by the
// per-sample weight, accumulate in fp32 (fp64 for fp32 tables) and write one D-wide pooled
// output row.  The pages' design is a Triton program per group of bags looping over the tables
// with four to eight row loads in flight; here a warp owns a work item of up to 32 consecutive
// bags of one table:
//   * the item's offsets come in with one coalesced load (lane k holds bag k's bounds), and
//     its ids stream through three 32-position register windows, two in use and one in
//     flight, so a bag's own critical path is only its row loads (offsets -> ids -> rows was
//     three dependent round trips per bag when each bag fetched its own ids);
//   * a row of D elements is split into 16-byte vectors; a group of next_pow2(vectors) lanes
//     covers one row, so one warp-wide load instruction fetches 32/group rows, and UNROLL such
//     instructions are issued before any is consumed (8 rows in flight per warp for fp16 D=128);
//   * unweighted 16-bit rows are added into the fp32 sums with the mixed-precision add of
//     sm_100+ (no separate widening instruction);
//   * the row groups are reduced with xor-shuffles and one group writes the fp32 result with
//     streaming 16-byte stores;
//   * one item per warp, CTAs launched table-major: the CTAs in flight read neighbouring parts of
//     the index array and mostly one table's rows, and an SM takes the next CTA as soon as one
//     retires (a resident grid-stride loop balanced uneven items worse: 3.1 vs 2.6 ms on the
//     83.9M-lookup stress batch).
// Out-of-range ids are repaired to row 0 in flight when fused bounds checking is on (writing
// the repaired id back), else skipped and counted; no id outside its table is dereferenced.
// The same kernel in dot mode computes the gradient with respect to the per-sample weights: the
// derivative of bag (t, b)'s pooled row with respect to psw[p] is W_t[idx[p]] (over L for mean
// pooling), so grad_psw[p] = <grad_out[b, table's columns], W_t[idx[p]]>; each lane holds its
// slice of the bag's gradient row and the row's dot product replaces its sum.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstring>
#include <mutex>

#include "tbe_internal.cuh"

namespace tbe {
namespace {

struct FwdArgs {
  const void* weights;
  const int64_t* woff;
  const int32_t* doff;
  const int64_t* roff;
  void* indices;
  const void* offsets;
  const float* psw;
  float* out;
  int64_t B;
  int64_t num_indices;
  int64_t unit_begin, unit_end;
  int64_t item_base;  // the launch's first work item
  int bags_per_item;  // 1..32
  int t_begin;        // first table of the launch (unit_begin / B)
  int64_t items_per_table, items;  // work items per table, in the launch
  int mean;           // mean pooling: the sum over the bag length (an empty bag stays 0)
  // dot mode (the gradient with respect to the per-sample weights): grad_out rows in, one fp32
  // per lookup out: grad_psw[p] = <grad_out[b, table's columns], W[idx[p]]> (/ L for mean)
  const float* grad;
  float* grad_psw;
  int total_D;
  int fused_bounds;
  unsigned long long* stats;
};

// The bytes of a CUtensorMap (a kernel parameter: 128 bytes, 64-byte aligned).
struct alignas(64) TmaMap {
  uint64_t w[16];
};
static_assert(sizeof(TmaMap) == sizeof(CUtensorMap), "tensor map size");

// Table (relative to the launch's first) of work item g: a 32-bit division when both fit.
__device__ __forceinline__ int64_t item_table(int64_t g, int64_t items_per_table) {
  if (((g | items_per_table) >> 31) == 0)
    return static_cast<uint32_t>(g) / static_cast<uint32_t>(items_per_table);
  return g / items_per_table;
}

__device__ __forceinline__ int next_pow2_int(int v) { return v <= 1 ? 1 : 1 << (32 - __clz(v - 1)); }

__device__ __forceinline__ void store_out(float* dst, const float (&v)[8]) {
  __stcs(reinterpret_cast<float4*>(dst), make_float4(v[0], v[1], v[2], v[3]));
  __stcs(reinterpret_cast<float4*>(dst) + 1, make_float4(v[4], v[5], v[6], v[7]));
}
__device__ __forceinline__ void store_out(float* dst, const float (&v)[4]) {
  __stcs(reinterpret_cast<float4*>(dst), make_float4(v[0], v[1], v[2], v[3]));
}

// Accumulate one raw vector of weights into fp32 (16-bit tables) or fp64 (fp32 tables).
// Unweighted 16-bit rows use the mixed-precision add of sm_100+ (an f16/bf16 operand added to
// an f32 accumulator in one instruction; the widening is exact, so the sum is the same as
// converting first and adding).
template <typename WT, int VB, bool PSW>
__device__ __forceinline__ void accumulate(typename VecIO<WT, VB>::Acc (&acc)[VecIO<WT, VB>::N],
                                           const typename VecIO<WT, VB>::Raw& v, float w) {
  using IO = VecIO<WT, VB>;
  using Acc = typename IO::Acc;
  constexpr int NE = IO::N;
  if constexpr (!PSW && sizeof(WT) == 2) {
    uint32_t words[IO::W];
    raw_words(v, words);
#pragma unroll
    for (int i = 0; i < IO::W; ++i) {
      if constexpr (std::is_same<WT, __half>::value) {
        asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
            "add.rn.f32.f16 %0, lo, %0;\n\tadd.rn.f32.f16 %1, hi, %1;\n\t}"
            : "+f"(acc[2 * i]), "+f"(acc[2 * i + 1])
            : "r"(words[i]));
      } else {
        asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
            "add.rn.f32.bf16 %0, lo, %0;\n\tadd.rn.f32.bf16 %1, hi, %1;\n\t}"
            : "+f"(acc[2 * i]), "+f"(acc[2 * i + 1])
            : "r"(words[i]));
      }
    }
  } else {
    float f[NE];
    IO::unpack(v, f);
#pragma unroll
    for (int i = 0; i < NE; ++i) {
      if (PSW) acc[i] += static_cast<Acc>(f[i]) * static_cast<Acc>(w);
      else acc[i] += static_cast<Acc>(f[i]);
    }
  }
}

// A 32-position window of the index stream, one position per lane: the row of the lookup
// (or -1 when it is skipped) and its per-sample weight.  Only positions in [lo, hi), the span of
// the lanes' own work item, are read; repairs (fused bounds) and counts happen here, so with
// monotone offsets each position of the stream is repaired or counted exactly once.
template <bool PSW> struct IdWindow {
  int32_t id;
  float w;
};

template <typename IT, bool PSW>
__device__ __forceinline__ IdWindow<PSW> load_window(const FwdArgs& a, int pos, int lo, int hi, int E) {
  IdWindow<PSW> r{-1, 0.0f};
  if (pos < lo || pos >= hi) return r;
  int64_t v = ld_int<IT>(a.indices, pos);
  bool ok = v >= 0 && v < E;
  if (PSW) r.w = __ldg(a.psw + pos);
  if (!ok) {
    if (a.fused_bounds) {
      static_cast<IT*>(a.indices)[pos] = IT(0);
      v = 0;
      ok = true;
      stat_add(a.stats, TBE_STAT_BAD_INDICES, 1);
    } else {
      stat_add(a.stats, TBE_STAT_UNREPAIRED, 1);
    }
  }
  r.id = ok ? static_cast<int32_t>(v) : -1;  // E < 2^31
  return r;
}

// Work item: up to 32 consecutive bags of one table (fewer when the batch is too small to give
// every warp several items).  A warp streams the item's part of the index
// array through three 32-position register windows (two in use, the third in flight), so the
// only loads on the critical path of a bag are its row loads: offsets and ids are fetched once
// per item and up to 64 positions ahead.  Offsets that are not monotone (not repaired) cost a
// reload of the windows where the stream jumps back or far ahead.
// DOT = the gradient with respect to the per-sample weights: the same walk over bags, windows and
// rows, but each lane keeps its slice of the bag's gradient row and every row is dotted into it
// (reduced within its row group) instead of being summed.
// Threads per CTA, and resident CTAs per SM for a 256-thread block (scaled to the block size).
// Two-warp CTAs: a CTA's slot frees as soon as its two items are done, so items of uneven
// length leave few warp slots idle (83.9M-lookup stress batch: 2.37 ms with 8-warp CTAs,
// 2.21 ms with 2-warp CTAs, 2.25 ms with 1-warp CTAs).
constexpr int kGatherThreads = 64;
template <typename WT, int MAXV>
constexpr int gather_min_blocks() {
  return (MAXV == 1 ? (sizeof(WT) == 4 ? 3 : 4) : (MAXV == 2 ? 2 : 1)) * (256 / kGatherThreads);
}

template <typename WT, typename IT, bool PSW, int VB, int MAXV, int UNROLL, bool DOT>
__global__ void __launch_bounds__(kGatherThreads, gather_min_blocks<WT, MAXV>())
fwd_gather_kernel(FwdArgs a) {
  using IO = VecIO<WT, VB>;
  using Raw = typename IO::Raw;
  using Acc = typename IO::Acc;
  constexpr int NE = IO::N;  // weight elements per vector
  const unsigned FULL = 0xffffffffu;
  const int lane = lane_id();
  const int K = a.bags_per_item;
  const int N = static_cast<int>(a.num_indices);
  // one work item per warp
  const int64_t g = a.item_base + ((static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5);
  if (g < a.items) {
    const int64_t tq = item_table(g, a.items_per_table);
    const int t = a.t_begin + static_cast<int>(tq);
    const int64_t b0 = (g - tq * a.items_per_table) * K;
    const int nb = static_cast<int>(min(static_cast<int64_t>(K), a.B - b0));
    const int64_t u0 = static_cast<int64_t>(t) * a.B + b0;
    const int col0 = __ldg(a.doff + t);
    const int D = __ldg(a.doff + t + 1) - col0;
    const int E = static_cast<int>(__ldg(a.roff + t + 1) - __ldg(a.roff + t));  // < 2^31
    const int nvec = D / NE;
    const int lpr = nvec >= kWarp ? kWarp : next_pow2_int(nvec);  // lanes per row (a power of 2)
    const int lpr_log = __ffs(lpr) - 1;
    const int rps_log = 5 - lpr_log;
    const int rps = 1 << rps_log;                                  // rows per load step
    const int slot = lane >> lpr_log;
    const int vi = lane & (lpr - 1);
    // row 0 of the table; this lane's vectors of a row (lanes past the row width re-read its last
    // vector in full batches: their sums are never stored); the item's first output row
    const Raw* table = reinterpret_cast<const Raw*>(static_cast<const WT*>(a.weights) + __ldg(a.woff + t));
    // this lane's vectors of row 0 as byte addresses: row id's vector m is at lbase[m] + id * rbytes,
    // one wide multiply-add
    const char* lbase[MAXV];
#pragma unroll
    for (int m = 0; m < MAXV; ++m) lbase[m] = reinterpret_cast<const char*>(table + min(vi + m * kWarp, nvec - 1));
    const uint32_t rbytes = static_cast<uint32_t>(nvec) * VB;
    auto at = [&](int m, int32_t id) {
      return reinterpret_cast<const Raw*>(lbase[m] + static_cast<uint64_t>(static_cast<uint32_t>(id)) * rbytes);
    };
    float* orow = a.out + b0 * a.total_D + col0 + vi * NE;
    const int qmax = min(UNROLL, lpr);  // a batch (qmax * rps rows) covers at most 32 positions

    // bag k of the item owns positions [s_k, e_k): lane k holds s_k in off_s and e_k in off_e
    int off_s = 0, off_e = 0;
    if (lane < nb) {
      off_s = static_cast<int>(clamp64(ld_int<IT>(a.offsets, u0 + lane), 0, N));
      off_e = static_cast<int>(clamp64(ld_int<IT>(a.offsets, u0 + lane + 1), off_s, N));
    }
    // span of the item's positions (the first s and last e unless offsets are not monotone)
    int lo = lane < nb ? off_s : N, hi = off_e;
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) {
      lo = min(lo, __shfl_xor_sync(FULL, lo, m));
      hi = max(hi, __shfl_xor_sync(FULL, hi, m));
    }
    int w0 = __shfl_sync(FULL, off_s, 0);
    IdWindow<PSW> wa = load_window<IT, PSW>(a, w0 + lane, lo, hi, E);
    IdWindow<PSW> wb = load_window<IT, PSW>(a, w0 + kWarp + lane, lo, hi, E);
    IdWindow<PSW> wc = load_window<IT, PSW>(a, w0 + 2 * kWarp + lane, lo, hi, E);

    for (int k = 0; k < nb; ++k) {
      const int s = __shfl_sync(FULL, off_s, k);
      const int e = __shfl_sync(FULL, off_e, k);
      Acc acc[MAXV][NE];  // the pooled sums; in DOT mode the bag's gradient row slice
      if constexpr (DOT) {
        const float* grow = a.grad + (b0 + k) * a.total_D + col0;
#pragma unroll
        for (int m = 0; m < MAXV; ++m)
#pragma unroll
          for (int i = 0; i < NE; ++i)
            acc[m][i] = vi + m * kWarp < nvec ? static_cast<Acc>(__ldg(grow + (vi + m * kWarp) * NE + i)) : Acc(0);
      } else {
#pragma unroll
        for (int m = 0; m < MAXV; ++m)
#pragma unroll
          for (int i = 0; i < NE; ++i) acc[m][i] = Acc(0);
      }
      const Acc inv_len = (DOT && a.mean && e > s) ? Acc(1) / static_cast<Acc>(e - s) : Acc(1);

      for (int c0 = s; c0 < e; c0 += kWarp) {  // 32 positions of the bag at a time
        // slide the windows so that c0 - w0 is in [0, 32) (warp-uniform)
        int rel0 = c0 - w0;
        if (rel0 >= kWarp && rel0 < 3 * kWarp) {
          while (rel0 >= kWarp) {
            wa = wb;
            wb = wc;
            wc = load_window<IT, PSW>(a, w0 + 3 * kWarp + lane, lo, hi, E);
            w0 += kWarp;
            rel0 -= kWarp;
          }
        } else if (rel0 < 0 || rel0 >= 3 * kWarp) {
          w0 = c0;
          rel0 = 0;
          wa = load_window<IT, PSW>(a, w0 + lane, lo, hi, E);
          wb = load_window<IT, PSW>(a, w0 + kWarp + lane, lo, hi, E);
          wc = load_window<IT, PSW>(a, w0 + 2 * kWarp + lane, lo, hi, E);
        }
        // lane l takes position c0 + l from the two windows in use
        const int rel = rel0 + lane;  // in [0, 64)
        const int32_t ida = __shfl_sync(FULL, wa.id, rel & (kWarp - 1));
        const int32_t idb = __shfl_sync(FULL, wb.id, rel & (kWarp - 1));
        const int n = min(kWarp, e - c0);
        const int32_t my_id = lane < n ? (rel < kWarp ? ida : idb) : -1;
        float my_w = 0.0f;  // 0 where no row is read, so a zero vector is never scaled by inf
        if (PSW) {
          const float pa = __shfl_sync(FULL, wa.w, rel & (kWarp - 1));
          const float pb = __shfl_sync(FULL, wb.w, rel & (kWarp - 1));
          if (my_id >= 0) my_w = rel < kWarp ? pa : pb;
        }
        const bool chunk_ok = __all_sync(FULL, lane >= n || my_id >= 0);  // no skipped id
        int j = 0;
        if constexpr (!DOT && !PSW) {  // (with weights the extra loop spills registers)
          if (chunk_ok && qmax == UNROLL) {
            // whole batches of valid rows first: unpredicated loads, no per-batch checks
            for (; j + rps * UNROLL <= n; j += rps * UNROLL) {
              Raw v[UNROLL][MAXV];
#pragma unroll
              for (int q = 0; q < UNROLL; ++q) {
                const int32_t id = __shfl_sync(FULL, my_id, j + q * rps + slot);
#pragma unroll
                for (int m = 0; m < MAXV; ++m) v[q][m] = ldg_raw(at(m, id));
              }
#pragma unroll
              for (int q = 0; q < UNROLL; ++q)
#pragma unroll
                for (int m = 0; m < MAXV; ++m) accumulate<WT, VB, false>(acc[m], v[q][m], 1.0f);
            }
          }
        }
        for (; j < n; j += rps * qmax) {  // the bag's last rows, batches with a skipped id, dot mode
          Raw v[UNROLL][MAXV];
          int nq = UNROLL;  // load steps of this batch that hold a row (warp-uniform)
          const bool full = chunk_ok && qmax == UNROLL && j + rps * UNROLL <= n;
          if (full) {
            // every row of the batch is valid: unpredicated loads
#pragma unroll
            for (int q = 0; q < UNROLL; ++q) {
              const int r = j + q * rps + slot;
              const int32_t id = __shfl_sync(FULL, my_id, r);
#pragma unroll
              for (int m = 0; m < MAXV; ++m) v[q][m] = ldg_raw(at(m, id));
            }
          } else {
            // the bag's last rows (or a batch with a skipped id): only the load steps that hold a
            // row are issued and summed
            nq = min(qmax, (n - j + rps - 1) >> rps_log);
#pragma unroll
            for (int q = 0; q < UNROLL; ++q) {
#pragma unroll
              for (int m = 0; m < MAXV; ++m) v[q][m] = Raw{};
              if (q < nq) {
                const int r = j + q * rps + slot;  // < 64; lanes past n hold -1
                const int32_t id = __shfl_sync(FULL, my_id, r & (kWarp - 1));
                const bool ok = r < n && id >= 0;
#pragma unroll
                for (int m = 0; m < MAXV; ++m)
                  if (ok && vi + m * kWarp < nvec) v[q][m] = ldg_raw(at(m, id));
              }
            }
          }
          if constexpr (DOT) {
            Acc dot[UNROLL];
#pragma unroll
            for (int q = 0; q < UNROLL; ++q) {
              dot[q] = 0;
#pragma unroll
              for (int m = 0; m < MAXV; ++m) {
                if (vi + m * kWarp < nvec) {  // lanes past the row width re-read its last vector
                  float f[NE];
                  IO::unpack(v[q][m], f);
#pragma unroll
                  for (int i = 0; i < NE; ++i) dot[q] += acc[m][i] * static_cast<Acc>(f[i]);
                }
              }
            }
            if (UNROLL == 4 && lpr >= 4) {
              // the four rows' partial dots reduced together: two halving rounds leave each lane
              // one row (the bits lpr/2 and lpr/4 of its lane pick which), then a plain xor
              // reduction over the remaining lanes of the row group
              const int o1 = lpr >> 1, o2 = lpr >> 2;
              const bool up1 = (lane & o1) != 0, up2 = (lane & o2) != 0;
              Acc k0 = up1 ? dot[2] : dot[0], k1 = up1 ? dot[3] : dot[1];
              k0 += __shfl_xor_sync(FULL, up1 ? dot[0] : dot[2], o1);
              k1 += __shfl_xor_sync(FULL, up1 ? dot[1] : dot[3], o1);
              Acc d = up2 ? k1 : k0;
              d += __shfl_xor_sync(FULL, up2 ? k0 : k1, o2);
              for (int off = o2 >> 1; off > 0; off >>= 1) d += __shfl_xor_sync(FULL, d, off);
              const int q = (up1 ? 2 : 0) + (up2 ? 1 : 0);
              const int r = j + q * rps + slot;
              if ((vi & (o2 - 1)) == 0 && q < qmax && r < n) a.grad_psw[c0 + r] = static_cast<float>(d * inv_len);
            } else {
#pragma unroll
              for (int q = 0; q < UNROLL; ++q) {
                Acc d = dot[q];
                for (int off = lpr >> 1; off > 0; off >>= 1) d += __shfl_xor_sync(FULL, d, off);
                const int r = j + q * rps + slot;
                if (vi == 0 && q < qmax && r < n) a.grad_psw[c0 + r] = static_cast<float>(d * inv_len);
              }
            }
          } else if (full) {
            // the weights are fetched here, after the loads, so they hold no registers meanwhile
#pragma unroll
            for (int q = 0; q < UNROLL; ++q) {
              const float wq = PSW ? __shfl_sync(FULL, my_w, j + q * rps + slot) : 1.0f;
#pragma unroll
              for (int m = 0; m < MAXV; ++m) accumulate<WT, VB, PSW>(acc[m], v[q][m], wq);
            }
          } else {
#pragma unroll
            for (int q = 0; q < UNROLL; ++q) {
              if (q < nq) {
                float wq = 1.0f;
                if (PSW) {
                  const int r = j + q * rps + slot;
                  wq = __shfl_sync(FULL, my_w, r & (kWarp - 1));
                  if (r >= n) wq = 0.0f;  // a row past the bag: its vector is zero
                }
#pragma unroll
                for (int m = 0; m < MAXV; ++m) accumulate<WT, VB, PSW>(acc[m], v[q][m], wq);
              }
            }
          }
        }
      }
      if constexpr (!DOT) {  // dot mode has no pooled row
        // reduce the row groups of the warp (lanes that share vi)
        for (int m = lpr; m < kWarp; m <<= 1) {
#pragma unroll
          for (int x = 0; x < MAXV; ++x)
#pragma unroll
            for (int i = 0; i < NE; ++i) acc[x][i] += __shfl_xor_sync(FULL, acc[x][i], m);
        }
        if (a.mean && e > s) {  // times 1 / L: within an ulp of the quotient, one division a bag
          const Acc inv = Acc(1) / static_cast<Acc>(e - s);
#pragma unroll
          for (int x = 0; x < MAXV; ++x)
#pragma unroll
            for (int i = 0; i < NE; ++i) acc[x][i] *= inv;
        }
        if (slot == 0) {
#pragma unroll
          for (int x = 0; x < MAXV; ++x) {
            if (vi + x * kWarp < nvec) {
              float o[NE];
#pragma unroll
              for (int i = 0; i < NE; ++i) o[i] = static_cast<float>(acc[x][i]);
              store_out(orow + x * kWarp * NE, o);
            }
          }
        }
        orow += a.total_D;
      }
    }
  }
}

// ------------------------------------------------------------------------------------------
// Row gather through the tensor memory accelerator (sm_100+): every table has the same width,
// so the packed weights are one [sum E, D] matrix and a tile::gather4 copy brings four of its
// rows (any four row numbers) into shared memory, completion counted in bytes on an mbarrier.
// A warp owns a work item of up to 32 consecutive bags, as in the register gather, and streams
// the item's lookups through a ring of kTmaStages four-row stages: lane 0 keeps the ring full
// (row numbers come from the same 32-position id windows, prefetched one window ahead), and
// the warp sums each row out of shared memory into the bag's fp32 accumulator, one row per
// step with each lane owning D/32 columns, so a finished bag needs no cross-lane reduction:
// the warp stores it as one coalesced row.  Up to 4 x kTmaStages rows per warp are in flight
// without holding registers (the register gather holds 8).  It is the TBE_GATHER_TMA option:
// on the 83.9M-lookup stress batch (256-byte rows, mostly L2 hits) it takes 3.1 ms against
// 2.1 ms for the register gather, whose instructions per lookup are fewer (23 against 30);
// on uniform ids over a 1M-row table (DRAM-bound) it is the faster one (0.048 vs 0.056 ms).
// Items whose offsets do not tile their span (possible only when the offsets were not
// repaired) take a plain per-bag loop instead.
// ------------------------------------------------------------------------------------------
constexpr int kTmaThreads = 64;
constexpr int kTmaWarps = kTmaThreads / kWarp;
constexpr int kTmaStages = 8;
constexpr int kTmaMinBlocks = 12;  // 16 KB of ring per CTA at D = 128
constexpr uint32_t kTmaWaitLimit = 1u << 22;

__device__ __forceinline__ void tma_gather4(void* dst, const TmaMap* map, int r0, int r1, int r2, int r3,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(0), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(smem_u32(bar))
      : "memory");
}

template <typename WT, int VB>
__device__ __forceinline__ typename VecIO<WT, VB>::Raw lds_raw(const uint8_t* p) {
  return *reinterpret_cast<const typename VecIO<WT, VB>::Raw*>(p);
}

// One bag's fp32 sums (NE columns per lane) to its output row; mean pooling divides by L.
template <int NE>
__device__ __forceinline__ void store_bag(float* orow, float (&acc)[NE], int len, bool mean) {
  if (mean && len > 0) {  // times 1 / L: within an ulp of the quotient, one division a bag
    const float inv = 1.0f / static_cast<float>(len);
#pragma unroll
    for (int i = 0; i < NE; ++i) acc[i] *= inv;
  }
  if constexpr (NE == 2) {
    __stcs(reinterpret_cast<float2*>(orow), make_float2(acc[0], acc[1]));
  } else {
    store_out(orow, acc);
  }
#pragma unroll
  for (int i = 0; i < NE; ++i) acc[i] = 0.0f;
}

template <typename WT, typename IT, bool PSW, int VB>
__global__ void __launch_bounds__(kTmaThreads, kTmaMinBlocks) fwd_tma_gather_kernel(
    const __grid_constant__ TmaMap tmap, FwdArgs a) {
  using IO = VecIO<WT, VB>;
  using Raw = typename IO::Raw;
  constexpr int NE = IO::N;          // columns per lane
  constexpr int RB = VB * kWarp;     // bytes per row (D = 32 * NE)
  constexpr int SB = 4 * RB;         // bytes per stage
  constexpr int S = kTmaStages;      // a power of 2, at most 8 (two id windows cover the ring)
  static_assert((S & (S - 1)) == 0 && S <= 8, "stage ring");
  const unsigned FULL = 0xffffffffu;
  extern __shared__ __align__(128) uint8_t s_ring[];  // [warp][stage][4 rows]
  __shared__ __align__(8) uint64_t s_bar[kTmaWarps][S];
  __shared__ __align__(16) int s_rows[kTmaWarps][2][kWarp];  // row numbers of two id windows
  __shared__ float s_psw[kTmaWarps][2][kWarp];               // their psw (weighted)
  __shared__ int s_mask[kTmaWarps][S];                        // bit j: row j of the stage is a lookup
  const int lane = lane_id(), wl = threadIdx.x / kWarp;
  uint8_t* ring = s_ring + wl * S * SB;
  uint64_t* bar = s_bar[wl];
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < S; ++s) mbar_init(&bar[s], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();

  const int K = a.bags_per_item;
  const int N = static_cast<int>(a.num_indices);
  const int64_t g = a.item_base + ((static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5);
  if (g >= a.items) return;
  const int64_t tq = item_table(g, a.items_per_table);
  const int t = a.t_begin + static_cast<int>(tq);
  const int64_t b0 = (g - tq * a.items_per_table) * K;
  const int nb = static_cast<int>(min(static_cast<int64_t>(K), a.B - b0));
  const int64_t u0 = static_cast<int64_t>(t) * a.B + b0;
  const int col0 = __ldg(a.doff + t);
  const int64_t rbase64 = __ldg(a.roff + t);
  const int E = static_cast<int>(__ldg(a.roff + t + 1) - rbase64);  // < 2^31
  const int rbase = static_cast<int>(rbase64);                     // sum E < 2^31
  float* orow0 = a.out + b0 * a.total_D + col0 + lane * NE;
  const bool mean = a.mean != 0;

  int off_s = 0, off_e = 0;
  if (lane < nb) {
    off_s = static_cast<int>(clamp64(ld_int<IT>(a.offsets, u0 + lane), 0, N));
    off_e = static_cast<int>(clamp64(ld_int<IT>(a.offsets, u0 + lane + 1), off_s, N));
  }
  int lo = lane < nb ? off_s : N, hi = off_e;
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) {
    lo = min(lo, __shfl_xor_sync(FULL, lo, m));
    hi = max(hi, __shfl_xor_sync(FULL, hi, m));
  }
  // do the bags tile [lo, hi) in order (always, once the offsets are repaired)?
  const int next_s = __shfl_down_sync(FULL, off_s, 1);
  const bool tiles = __all_sync(FULL, lane >= nb - 1 || off_e == next_s);
  float acc[NE];
#pragma unroll
  for (int i = 0; i < NE; ++i) acc[i] = 0.0f;

  if (!tiles) {
    // plain per-bag walk: ids through one window per 32 positions, rows by direct loads
    const Raw* table = reinterpret_cast<const Raw*>(static_cast<const WT*>(a.weights) + __ldg(a.woff + t));
    for (int k = 0; k < nb; ++k) {
      const int s = __shfl_sync(FULL, off_s, k), e = __shfl_sync(FULL, off_e, k);
      for (int c0 = s; c0 < e; c0 += kWarp) {
        const IdWindow<PSW> w = load_window<IT, PSW>(a, c0 + lane, s, e, E);
        const int n = min(kWarp, e - c0);
        for (int r = 0; r < n; ++r) {
          const int32_t id = __shfl_sync(FULL, w.id, r);
          const float wr = PSW ? __shfl_sync(FULL, w.w, r) : 1.0f;
          if (id >= 0) accumulate<WT, VB, PSW>(acc, ldg_raw(table + static_cast<int64_t>(id) * kWarp + lane), wr);
        }
      }
      store_bag<NE>(orow0 + static_cast<int64_t>(k) * a.total_D, acc, e - s, mean);
    }
    return;
  }

  // Producer.  Stage i holds positions lo + 4i .. lo + 4i + 3; id window m (positions
  // lo + 32m .. +31, stages 8m .. 8m + 7) is turned into row numbers (the table's row 0 where a
  // lookup is skipped or past hi) and a validity mask by the whole warp, one position per lane,
  // into shared slot m & 1, while window m + 1's ids are already on their way.  Lane 0 then
  // issues a stage with one 16-byte read of four row numbers.
  const int nst = (hi - lo + 3) >> 2;
  IdWindow<PSW> pre = load_window<IT, PSW>(a, lo + lane, lo, hi, E);
  uint32_t wbits = 0;  // validity of the producer's current window
  auto stage_window = [&](int m) {
    const IdWindow<PSW> cur = pre;
    pre = load_window<IT, PSW>(a, lo + (m + 1) * kWarp + lane, lo, hi, E);
    const bool ok = cur.id >= 0;  // false past hi (the window reads nothing there)
    s_rows[wl][m & 1][lane] = rbase + (ok ? cur.id : 0);
    if (PSW) s_psw[wl][m & 1][lane] = cur.w;
    wbits = __ballot_sync(FULL, ok);
    __syncwarp();
  };
  int issued = 0;
  auto issue = [&]() {
    if ((issued & 7) == 0) stage_window(issued >> 3);
    const int slot = issued & (S - 1);
    const int r = (issued & 7) * 4;
    if (lane == 0) {
      const int4 rows = *reinterpret_cast<const int4*>(&s_rows[wl][(issued >> 3) & 1][r]);
      s_mask[wl][slot] = static_cast<int>((wbits >> r) & 0xFu);
      fence_proxy_async_smem();  // the slot's earlier reads before the copy overwrites it
      mbar_arrive_expect_tx(&bar[slot], SB);
      tma_gather4(ring + slot * SB, &tmap, rows.x, rows.y, rows.z, rows.w, &bar[slot]);
    }
    ++issued;
  };

  // bags before the first row (empty ones) are written as zeros
  int k = 0;
  int s_k = __shfl_sync(FULL, off_s, 0), e_k = __shfl_sync(FULL, off_e, 0);
  auto next_bag = [&]() {  // store bag k, then move to the next non-empty bag (storing empty ones)
    store_bag<NE>(orow0 + static_cast<int64_t>(k) * a.total_D, acc, e_k - s_k, mean);
    ++k;
    while (k < nb) {
      s_k = __shfl_sync(FULL, off_s, k);
      e_k = __shfl_sync(FULL, off_e, k);
      if (e_k > s_k) break;
      store_bag<NE>(orow0 + static_cast<int64_t>(k) * a.total_D, acc, 0, mean);
      ++k;
    }
  };
  if (e_k == s_k) next_bag();  // a leading empty bag (stored as zeros)
  while (issued < nst && issued < S) issue();
  __syncwarp();

  bool failed = false;
  int i = 0;
  for (; i < nst; ++i) {
    const int slot = i & (S - 1);
    if (!mbar_wait_bounded(&bar[slot], (i / S) & 1, kTmaWaitLimit)) {
      failed = true;
      if (lane == 0) stat_add(a.stats, TBE_STAT_WAIT_TIMEOUT, 1);
      break;
    }
    const uint8_t* st = ring + slot * SB + lane * VB;
    const int p0 = lo + 4 * i;
    const int mask = s_mask[wl][slot];
    const float* wv = &s_psw[wl][(i >> 3) & 1][(i & 7) * 4];
    if (mask == 0xF && e_k >= p0 + 4) {
      // four lookups of bag k
      Raw v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) v[j] = lds_raw<WT, VB>(st + j * RB);
#pragma unroll
      for (int j = 0; j < 4; ++j) accumulate<WT, VB, PSW>(acc, v[j], PSW ? wv[j] : 1.0f);
      if (e_k == p0 + 4) next_bag();
    } else {
      const int n = min(4, hi - p0);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (j < n) {
          if (mask & (1 << j)) accumulate<WT, VB, PSW>(acc, lds_raw<WT, VB>(st + j * RB), PSW ? wv[j] : 1.0f);
          if (p0 + j + 1 == e_k) next_bag();
        }
      }
    }
    __syncwarp();  // every lane has read the slot (and the window entries of the stage)
    if (issued < nst) {
      issue();
      __syncwarp();
    }
  }
  if (failed) {
    // a copy that never signalled: wait once more (bounded) for every stage still in flight
    // before the warp's shared memory can be released
    for (int q = i; q < issued; ++q) mbar_wait_bounded(&bar[q & (S - 1)], (q / S) & 1, kTmaWaitLimit);
  }
}

// ------------------------------------------------------------------------------------------
// Very long bags of 16-bit tables, summed again in segments.  The gathers above keep one fp32
// running sum per lane over a whole bag, which is all the fp32 accumulation the pages prescribe
// needs for ordinary bags; but a bag of 10^5 - 10^6 lookups of a few hot rows adds the same value
// into one fp32 sum 10^5 times, each addition rounding the same way, and drifts by about 2e-3 of
// the sum (at kLongBag = 16384 lookups the same drift is under 1e-4).  This pass finds the bags
// longer than kLongBag lookups and writes their output rows again from sums of kSegment-lookup
// segments, each segment summed in fp32 and the segment sums added in fp32, which keeps the error
// near (kSegment + L / kSegment) roundings.  It runs after the gather (and after the counts x
// table path, whose scalar tail past the 256th id also sums sequentially), reads ids the forward
// has already repaired (skipping out-of-range ones without counting them: the gather counted
// them), and leaves every other bag alone: for batches without such bags it costs one coalesced
// read of the offsets (the bag walk is a rare path, kept out of the scan's registers).
// ------------------------------------------------------------------------------------------
constexpr int kLongBag = 16384;
constexpr int kSegment = 1024;
constexpr int kLongThreads = 128;

template <typename WT, typename IT, bool PSW, int VB>
__global__ void __launch_bounds__(kLongThreads, 8) fwd_long_bags_kernel(FwdArgs a) {
  using IO = VecIO<WT, VB>;  // rows read as 16-byte vectors, or 8-byte ones for widths that need it
  using Raw = typename IO::Raw;
  constexpr int NE = IO::N;
  constexpr int UNROLL = PSW ? 4 : 8;
  const unsigned FULL = 0xffffffffu;
  const int lane = lane_id();
  const int N = static_cast<int>(a.num_indices);
  const int64_t units = a.unit_end - a.unit_begin;
  const int64_t warp0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int64_t warps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t base = warp0 * kWarp; base < units; base += warps * kWarp) {
    const int64_t u = a.unit_begin + base + lane;
    int s = 0, e = 0;
    if (base + lane < units) {
      s = static_cast<int>(clamp64(ld_int<IT>(a.offsets, u), 0, N));
      e = static_cast<int>(clamp64(ld_int<IT>(a.offsets, u + 1), s, N));
    }
    unsigned m = __ballot_sync(FULL, e - s > kLongBag);
    while (m != 0) {
      const int j = __ffs(m) - 1;
      m &= m - 1;
      const int64_t ub = a.unit_begin + base + j;
      const int bs = __shfl_sync(FULL, s, j), be = __shfl_sync(FULL, e, j);
      const int t = static_cast<int>(ub / a.B);
      const int64_t b = ub - static_cast<int64_t>(t) * a.B;
      const int col0 = __ldg(a.doff + t);
      const int nvec = (__ldg(a.doff + t + 1) - col0) * static_cast<int>(sizeof(WT)) / VB;
      const int E = static_cast<int>(__ldg(a.roff + t + 1) - __ldg(a.roff + t));
      const Raw* table = reinterpret_cast<const Raw*>(static_cast<const WT*>(a.weights) + __ldg(a.woff + t));
      const int lpr = nvec >= kWarp ? kWarp : (nvec <= 1 ? 1 : 1 << (32 - __clz(nvec - 1)));
      const int rps = kWarp / lpr, slot = lane / lpr, vi = lane % lpr;
      const float inv = a.mean ? 1.0f / static_cast<float>(be - bs) : 1.0f;
      float* orow = a.out + b * a.total_D + col0;
      // one pass over the bag per 32 vectors of the row (one pass for rows of up to 32 * VB bytes)
      for (int c = vi; c - vi < nvec; c += kWarp) {
        float tot[NE], seg[NE];
#pragma unroll
        for (int i = 0; i < NE; ++i) tot[i] = seg[i] = 0.0f;
        for (int g0 = bs; g0 < be; g0 += kSegment) {
          const int g1 = be - g0 > kSegment ? g0 + kSegment : be;
          for (int p = g0; p < g1; p += rps * UNROLL) {
            Raw v[UNROLL];
            float w[UNROLL];
#pragma unroll
            for (int q = 0; q < UNROLL; ++q) {
              const int pos = p + q * rps + slot;  // this slot's row of load step q
              int64_t id = -1;
              w[q] = 0.0f;
              if (pos < g1) {
                id = ld_int<IT>(a.indices, pos);
                if (id < 0 || id >= E) id = -1;  // skipped (and counted) by the gather
                else if (PSW) w[q] = __ldg(a.psw + pos);
              }
              v[q] = Raw{};
              if (id >= 0 && c < nvec) v[q] = ldg_raw(table + id * nvec + c);
            }
#pragma unroll
            for (int q = 0; q < UNROLL; ++q) {
              float f[NE];
              IO::unpack(v[q], f);
#pragma unroll
              for (int i = 0; i < NE; ++i) seg[i] += PSW ? f[i] * w[q] : f[i];
            }
          }
          // the segment's sum over the row slots, added into the bag's total
#pragma unroll
          for (int i = 0; i < NE; ++i) {
            float v = seg[i];
            for (int o = lpr; o < kWarp; o <<= 1) v += __shfl_xor_sync(FULL, v, o);
            tot[i] += v;
            seg[i] = 0.0f;
          }
        }
        if (slot == 0 && c < nvec) {
#pragma unroll
          for (int i = 0; i < NE; ++i) tot[i] *= inv;
          store_out(orow + c * NE, tot);
        }
      }
    }
  }
}

// Bags per work item: about eight items per resident warp, at most 32 bags each.
inline int bags_per_item_for(int64_t tables, int64_t B, int64_t warps) {
  const int64_t per_item = tables * B / (8 * warps);
  return per_item < 1 ? 1 : (per_item > kWarp ? kWarp : static_cast<int>(per_item));
}

template <typename WT, typename IT, bool PSW, int VB, int MAXV>
cudaError_t launch_t(const FwdArgs& a, const DeviceInfo& dev, cudaStream_t s) {
  constexpr int UNROLL = MAXV >= 4 ? 1 : (MAXV == 2 ? 2 : 4);  // 4 to 8 loads in flight per lane
  // the gradient with respect to psw does not read psw: it runs the unweighted walk in DOT mode
  auto k = a.grad_psw != nullptr ? fwd_gather_kernel<WT, IT, false, VB, MAXV, UNROLL, true>
                                 : fwd_gather_kernel<WT, IT, PSW, VB, MAXV, UNROLL, false>;
  const int threads = kGatherThreads;
  const int64_t tables = (a.unit_end - a.unit_begin) / a.B;
  const int64_t warps = static_cast<int64_t>(persistent_grid(k, threads, 0, dev, INT64_MAX)) * (threads / kWarp);
  // about eight items per warp, at most 32 bags per item
  FwdArgs ak = a;
  ak.bags_per_item = bags_per_item_for(tables, a.B, warps);
  ak.t_begin = static_cast<int>(a.unit_begin / a.B);
  ak.items_per_table = (a.B + ak.bags_per_item - 1) / ak.bags_per_item;
  const int64_t items = tables * ak.items_per_table;
  ak.items = items;
  // One item per warp: CTAs retire as their items finish and the block scheduler hands the SM
  // to the next one, which balances items of uneven length better than a resident grid-stride
  // loop.  Past the launch's grid limit the items go out in several launches.
  constexpr int64_t kMaxGrid = 0x7fffffff;
  const int64_t per_launch = kMaxGrid * (threads / kWarp);
  for (int64_t base = 0; base < items; base += per_launch) {
    const int64_t n = items - base < per_launch ? items - base : per_launch;
    ak.item_base = base;
    k<<<static_cast<unsigned>((n + (threads / kWarp) - 1) / (threads / kWarp)), threads, 0, s>>>(ak);
    note_launch();
  }
  return cudaGetLastError();
}

template <typename WT, typename IT, bool PSW, int VB>
cudaError_t launch_tma_t(const FwdArgs& a, const TmaMap& map, const DeviceInfo& dev, cudaStream_t s) {
  auto k = fwd_tma_gather_kernel<WT, IT, PSW, VB>;
  const size_t smem = static_cast<size_t>(kTmaWarps) * kTmaStages * 4 * VB * kWarp;
  if (smem > 48 * 1024) {
    static std::atomic<uint64_t> attr_set{0};
    const uint64_t bit = uint64_t(1) << (dev.id & 63);
    if ((attr_set.load() & bit) == 0) {
      const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
      if (e != cudaSuccess) return e;
      attr_set.fetch_or(bit);
    }
  }
  const int64_t tables = (a.unit_end - a.unit_begin) / a.B;
  const int64_t warps = static_cast<int64_t>(persistent_grid(k, kTmaThreads, smem, dev, INT64_MAX)) * kTmaWarps;
  FwdArgs ak = a;
  ak.bags_per_item = bags_per_item_for(tables, a.B, warps);
  ak.t_begin = static_cast<int>(a.unit_begin / a.B);
  ak.items_per_table = (a.B + ak.bags_per_item - 1) / ak.bags_per_item;
  const int64_t items = tables * ak.items_per_table;
  ak.items = items;
  constexpr int64_t kMaxGrid = 0x7fffffff;
  const int64_t per_launch = kMaxGrid * kTmaWarps;
  for (int64_t base = 0; base < items; base += per_launch) {
    const int64_t n = items - base < per_launch ? items - base : per_launch;
    ak.item_base = base;
    k<<<static_cast<unsigned>((n + kTmaWarps - 1) / kTmaWarps), kTmaThreads, smem, s>>>(map, ak);
    note_launch();
  }
  return cudaGetLastError();
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link against libcuda).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// The packed weights of equal-width tables as one [rows, D] matrix of 16-bit elements whose
// copy box is one row: the tensor map of the tile::gather4 loads.
bool encode_row_map(TmaMap* out, const void* weights, int64_t rows, int D, int wdtype) {
  const PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (encode == nullptr) return false;
  CUtensorMap m;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(D) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(D), 1};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = encode(&m, wdtype == TBE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                            2, const_cast<void*>(weights), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  std::memcpy(out, &m, sizeof(m));
  return true;
}

template <typename WT, typename IT, bool PSW>
cudaError_t dispatch_tma(const FwdArgs& a, const TmaMap& map, int D, const DeviceInfo& dev, cudaStream_t s) {
  switch (D) {
    case 64: return launch_tma_t<WT, IT, PSW, 4>(a, map, dev, s);
    case 128: return launch_tma_t<WT, IT, PSW, 8>(a, map, dev, s);
    default: return launch_tma_t<WT, IT, PSW, 16>(a, map, dev, s);
  }
}

template <typename WT, typename IT, bool PSW, int VB>
cudaError_t dispatch_maxv(const FwdArgs& a, int maxv, const DeviceInfo& dev, cudaStream_t s) {
  switch (maxv) {
    case 1: return launch_t<WT, IT, PSW, VB, 1>(a, dev, s);
    case 2: return launch_t<WT, IT, PSW, VB, 2>(a, dev, s);
    case 4: return launch_t<WT, IT, PSW, VB, 4>(a, dev, s);
    default: return launch_t<WT, IT, PSW, VB, 8>(a, dev, s);
  }
}

template <typename WT, typename IT, bool PSW>
cudaError_t dispatch_vb(const FwdArgs& a, int vb, int maxv, const DeviceInfo& dev, cudaStream_t s) {
  if constexpr (sizeof(WT) == 4) {
    return dispatch_maxv<WT, IT, PSW, 16>(a, maxv, dev, s);
  } else {
    if (vb == 16) return dispatch_maxv<WT, IT, PSW, 16>(a, maxv, dev, s);
    return dispatch_maxv<WT, IT, PSW, 8>(a, maxv, dev, s);
  }
}

template <typename WT>
cudaError_t dispatch_it(const FwdArgs& a, int itype, bool psw, int vb, int maxv,
                        const DeviceInfo& dev, cudaStream_t s) {
  if (itype == TBE_I32) {
    return psw ? dispatch_vb<WT, int32_t, true>(a, vb, maxv, dev, s)
               : dispatch_vb<WT, int32_t, false>(a, vb, maxv, dev, s);
  }
  return psw ? dispatch_vb<WT, int64_t, true>(a, vb, maxv, dev, s)
             : dispatch_vb<WT, int64_t, false>(a, vb, maxv, dev, s);
}

}  // namespace

// The TMA row gather takes 16-bit tables of one width D in {64, 128, 256} (the packed weights
// are then one [sum E, D] matrix; a row is 32 lanes x D/32 elements).
bool tma_gather_eligible(const Problem& P) {
  if (P.wbytes != 2 || P.T == 0) return false;
  for (int t = 0; t < P.T; ++t)
    if (P.D[t] != P.max_D) return false;
  return P.max_D == 64 || P.max_D == 128 || P.max_D == 256;
}

cudaError_t launch_forward_gather(const Problem& P, const tbe_tables& tab, const void* weights,
                                  void* indices, const void* offsets, const float* psw, float* out,
                                  int64_t unit_begin, int64_t unit_end, bool fused_bounds, bool allow_tma,
                                  unsigned long long* stats, const DeviceInfo& dev, cudaStream_t s) {
  if (unit_end <= unit_begin) return cudaSuccess;
  FwdArgs a;
  a.weights = weights;
  a.woff = tab.weight_offsets;
  a.doff = tab.D_offsets;
  a.roff = tab.row_offsets;
  a.indices = indices;
  a.offsets = offsets;
  a.psw = psw;
  a.out = out;
  a.B = P.B;
  a.num_indices = P.num_indices;
  a.unit_begin = unit_begin;
  a.item_base = 0;
  a.unit_end = unit_end;
  a.total_D = P.total_D;
  a.fused_bounds = fused_bounds ? 1 : 0;
  a.mean = P.pooling == TBE_POOL_MEAN;
  a.grad = nullptr;
  a.grad_psw = nullptr;
  a.stats = stats;
  const bool has_psw = psw != nullptr;
  if (allow_tma && tma_gather_eligible(P)) {
    TmaMap map;
    if (encode_row_map(&map, weights, P.total_rows, P.max_D, P.wdtype)) {
      if (P.wdtype == TBE_F16) {
        if (P.itype == TBE_I32)
          return has_psw ? dispatch_tma<__half, int32_t, true>(a, map, P.max_D, dev, s)
                         : dispatch_tma<__half, int32_t, false>(a, map, P.max_D, dev, s);
        return has_psw ? dispatch_tma<__half, int64_t, true>(a, map, P.max_D, dev, s)
                       : dispatch_tma<__half, int64_t, false>(a, map, P.max_D, dev, s);
      }
      if (P.itype == TBE_I32)
        return has_psw ? dispatch_tma<__nv_bfloat16, int32_t, true>(a, map, P.max_D, dev, s)
                       : dispatch_tma<__nv_bfloat16, int32_t, false>(a, map, P.max_D, dev, s);
      return has_psw ? dispatch_tma<__nv_bfloat16, int64_t, true>(a, map, P.max_D, dev, s)
                     : dispatch_tma<__nv_bfloat16, int64_t, false>(a, map, P.max_D, dev, s);
    }
  }
  const int vb = P.vec_bytes;
  const int ne = vb / P.wbytes;
  const int max_nvec = P.max_D / ne;
  int maxv = (max_nvec + kWarp - 1) / kWarp;
  maxv = maxv <= 1 ? 1 : (maxv <= 2 ? 2 : (maxv <= 4 ? 4 : 8));
  switch (P.wdtype) {
    case TBE_F32: return dispatch_it<float>(a, P.itype, has_psw, vb, maxv, dev, s);
    case TBE_F16: return dispatch_it<__half>(a, P.itype, has_psw, vb, maxv, dev, s);
    default: return dispatch_it<__nv_bfloat16>(a, P.itype, has_psw, vb, maxv, dev, s);
  }
}

// Long bags of 16-bit tables in units [unit_begin, unit_end), summed again in segments (see
// fwd_long_bags_kernel); fp32 tables sum in fp64 and need no second pass.
cudaError_t launch_forward_long_bags(const Problem& P, const tbe_tables& tab, const void* weights,
                                     const void* indices, const void* offsets, const float* psw, float* out,
                                     int64_t unit_begin, int64_t unit_end, const DeviceInfo& dev, cudaStream_t s) {
  if (unit_end <= unit_begin || P.wbytes != 2) return cudaSuccess;
  if (P.num_indices <= kLongBag) return cudaSuccess;  // no bag can be long
  FwdArgs a{};
  a.weights = weights;
  a.woff = tab.weight_offsets;
  a.doff = tab.D_offsets;
  a.roff = tab.row_offsets;
  a.indices = const_cast<void*>(indices);  // read only
  a.offsets = offsets;
  a.psw = psw;
  a.out = out;
  a.B = P.B;
  a.num_indices = P.num_indices;
  a.unit_begin = unit_begin;
  a.unit_end = unit_end;
  a.total_D = P.total_D;
  a.mean = P.pooling == TBE_POOL_MEAN;
  const int64_t warps_needed = (unit_end - unit_begin + kWarp - 1) / kWarp;
  int64_t blocks = (warps_needed + (kLongThreads / kWarp) - 1) / (kLongThreads / kWarp);
  const int64_t cap = static_cast<int64_t>(dev.sms) * 8;
  if (blocks > cap) blocks = cap;
  const bool w = psw != nullptr;
  const bool i32 = P.itype == TBE_I32;
  auto go = [&](auto wt, auto vb) {
    using WT = decltype(wt);
    constexpr int VB = decltype(vb)::value;
    if (i32) w ? fwd_long_bags_kernel<WT, int32_t, true, VB><<<blocks, kLongThreads, 0, s>>>(a)
             : fwd_long_bags_kernel<WT, int32_t, false, VB><<<blocks, kLongThreads, 0, s>>>(a);
    else w ? fwd_long_bags_kernel<WT, int64_t, true, VB><<<blocks, kLongThreads, 0, s>>>(a)
           : fwd_long_bags_kernel<WT, int64_t, false, VB><<<blocks, kLongThreads, 0, s>>>(a);
  };
  using V16 = std::integral_constant<int, 16>;
  using V8 = std::integral_constant<int, 8>;
  if (P.wdtype == TBE_F16) {
    if (P.vec_bytes == 16) go(__half{}, V16{});
    else go(__half{}, V8{});
  } else {
    if (P.vec_bytes == 16) go(__nv_bfloat16{}, V16{});
    else go(__nv_bfloat16{}, V8{});
  }
  note_launch();
  return cudaGetLastError();
}

// The gradient with respect to the per-sample weights: the gather's walk in dot mode over every
// table (it neither repairs nor counts ids: the forward did).
cudaError_t launch_psw_gradient(const Problem& P, const tbe_tables& tab, const void* weights,
                                const void* indices, const void* offsets, const float* grad_out,
                                float* grad_psw, const DeviceInfo& dev, cudaStream_t s) {
  if (P.TB == 0 || P.num_indices == 0) return cudaSuccess;
  FwdArgs a;
  a.weights = weights;
  a.woff = tab.weight_offsets;
  a.doff = tab.D_offsets;
  a.roff = tab.row_offsets;
  a.indices = const_cast<void*>(indices);  // read only: fused_bounds is off
  a.offsets = offsets;
  a.psw = nullptr;
  a.out = nullptr;
  a.B = P.B;
  a.num_indices = P.num_indices;
  a.unit_begin = 0;
  a.item_base = 0;
  a.unit_end = P.TB;
  a.total_D = P.total_D;
  a.fused_bounds = 0;
  a.mean = P.pooling == TBE_POOL_MEAN;
  a.grad = grad_out;
  a.grad_psw = grad_psw;
  a.stats = nullptr;
  const int vb = P.vec_bytes;
  const int ne = vb / P.wbytes;
  const int max_nvec = P.max_D / ne;
  int maxv = (max_nvec + kWarp - 1) / kWarp;
  maxv = maxv <= 1 ? 1 : (maxv <= 2 ? 2 : (maxv <= 4 ? 4 : 8));
  switch (P.wdtype) {
    case TBE_F32: return dispatch_it<float>(a, P.itype, false, vb, maxv, dev, s);
    case TBE_F16: return dispatch_it<__half>(a, P.itype, false, vb, maxv, dev, s);
    default: return dispatch_it<__nv_bfloat16>(a, P.itype, false, vb, maxv, dev, s);
  }
}

}  // namespace tbe
