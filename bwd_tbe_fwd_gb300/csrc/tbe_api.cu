// tbe_api.cu -- the C interface (tbe.h): argument validation, the host-side plan of each call
// (sizes only from the host description, never from device data), workspace carving and the
// launch sequence of each operation.  Nothing here synchronizes with the device, copies device
// data to the host, or allocates memory.
#include <algorithm>
#include <cstring>
#include <mutex>

#include <nvtx3/nvToolsExt.h>

#include "tbe_internal.cuh"

namespace tbe {

namespace {
thread_local int g_last_cuda_error = 0;
thread_local int64_t g_launches = 0;

// Adds the launches of the current call to the caller's host counter, if any.
struct LaunchTally {
  const tbe_options& o;
  explicit LaunchTally(const tbe_options& opt) : o(opt) { g_launches = 0; }
  ~LaunchTally() {
    if (o.launch_counter != nullptr) *o.launch_counter += g_launches;
  }
};

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int bucket_of(int D) {
  int k = 0;
  while ((1 << k) < D) ++k;
  return k;
}

// NVTX range names: event i ends stage i and begins stage i + 1 (event 0 begins stage 1).
const char* const kFwdRanges[TBE_FWD_NUM_EVENTS] = {"tbe_forward", "tbe_forward.gather", "tbe_forward.histogram"};
const char* const kBwdRanges[TBE_BWD_NUM_EVENTS] = {
    "tbe_backward",         "tbe_backward.expand", "tbe_backward.sort",  "tbe_backward.rle",
    "tbe_backward.classify", "tbe_backward.short",  "tbe_backward.long", "tbe_backward.apply",
    "tbe_backward.histogram"};
thread_local int g_nvtx_open = 0;  // ranges this thread has pushed and not yet popped

// Records stage-boundary event i (if the caller asked for events) and, with opt.nvtx, closes the
// NVTX range of the stage that ends here and opens the next one.
void record(const tbe_options& opt, int i, cudaStream_t s, const char* const* names, int n) {
  if (opt.events != nullptr && i < opt.num_events && opt.events[i] != nullptr)
    cudaEventRecord(static_cast<cudaEvent_t>(opt.events[i]), s);
  if (opt.nvtx) {
    if (i > 0 && g_nvtx_open > 0) {
      nvtxRangePop();
      --g_nvtx_open;
    }
    if (i + 1 < n) {
      nvtxRangePushA(names[i + 1]);
      ++g_nvtx_open;
    }
  }
}
void record(const tbe_options& opt, int i, cudaStream_t s) {  // backward stages
  record(opt, i, s, kBwdRanges, TBE_BWD_NUM_EVENTS);
}
void record_fwd(const tbe_options& opt, int i, cudaStream_t s) {
  record(opt, i, s, kFwdRanges, TBE_FWD_NUM_EVENTS);
}

// Closes the NVTX ranges a call left open (it returned early on an error).
struct RangeGuard {
  ~RangeGuard() {
    for (; g_nvtx_open > 0; --g_nvtx_open) nvtxRangePop();
  }
};

tbe_options resolve(const tbe_options* opt) {
  tbe_options o;
  tbe_default_options(&o);
  if (opt != nullptr) o = *opt;
  return o;
}

tbe_status check_options(const tbe_options& o) {
  if (o.long_threshold < 1 || o.chunk < 1) return TBE_ERR_INVALID_ARG;
  if (o.long_mode < TBE_LONG_AUTO || o.long_mode > TBE_LONG_FUSED) return TBE_ERR_INVALID_ARG;
  if (o.scheduler != TBE_SCHED_GRID && o.scheduler != TBE_SCHED_PERSISTENT && o.scheduler != TBE_SCHED_CLC)
    return TBE_ERR_INVALID_ARG;
  if (o.merge != TBE_MERGE_ATOMIC && o.merge != TBE_MERGE_BULK) return TBE_ERR_INVALID_ARG;
  if (o.gather != TBE_GATHER_REGISTER && o.gather != TBE_GATHER_TMA) return TBE_ERR_INVALID_ARG;
  if (o.num_events < 0 || (o.num_events > 0 && o.events == nullptr)) return TBE_ERR_INVALID_ARG;
  if (o.classify_mode != TBE_CLASSIFY_ORDERED && o.classify_mode != TBE_CLASSIFY_ATOMIC) return TBE_ERR_INVALID_ARG;
  if (o.prepared != 0 && o.prepared != 1) return TBE_ERR_INVALID_ARG;
  if (!aligned(o.forward_ws, 16)) return TBE_ERR_INVALID_ARG;
  return TBE_OK;
}

// The counts x table tables whose per-bag counts the forward saves in its workspace (the first
// kMaxHistTables eligible ones, as the backward takes them): their count and the bytes.
int saved_count_tables(const Problem& P, const tbe_options& o) {
  int n = 0;
  for (int t = 0; t < P.T && n < kMaxHistTables; ++t) n += hist_forward_eligible(P, o, t) ? 1 : 0;
  return n;
}
}  // namespace

tbe_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return TBE_OK;
  g_last_cuda_error = static_cast<int>(e);
  return TBE_ERR_CUDA;
}

void note_launch(int n) { g_launches += n; }

tbe_status make_problem(const tbe_problem* p, Problem* out) {
  if (p == nullptr || out == nullptr) return TBE_ERR_INVALID_ARG;
  if (p->T < 1 || p->B < 0 || p->num_indices < 0 || p->D == nullptr || p->E == nullptr)
    return TBE_ERR_INVALID_ARG;
  if (p->T > kMaxTables) return TBE_ERR_UNSUPPORTED;
  if (p->wdtype != TBE_F32 && p->wdtype != TBE_F16 && p->wdtype != TBE_BF16) return TBE_ERR_UNSUPPORTED;
  if (p->itype != TBE_I32 && p->itype != TBE_I64) return TBE_ERR_UNSUPPORTED;
  if (p->pooling != TBE_POOL_SUM && p->pooling != TBE_POOL_MEAN) return TBE_ERR_INVALID_ARG;
  Problem& P = *out;
  P = Problem();
  P.T = p->T;
  P.B = p->B;
  P.TB = static_cast<int64_t>(p->T) * p->B;
  P.num_indices = p->num_indices;
  P.wdtype = p->wdtype;
  P.itype = p->itype;
  P.weighted = p->weighted != 0;
  P.pooling = p->pooling;
  // weighted problems carry psw (over L for mean pooling) through the sort; unweighted mean
  // pooling needs only 1 / L, which the update kernels take from the offsets by the bag id
  P.scaled = P.weighted;
  P.mean_inv = !P.weighted && P.pooling == TBE_POOL_MEAN;
  P.wbytes = p->wdtype == TBE_F32 ? 4 : 2;
  P.D.assign(p->D, p->D + p->T);
  P.E.assign(p->E, p->E + p->T);
  P.long_bags.assign(p->T, 0);
  if (p->long_bags != nullptr) P.long_bags.assign(p->long_bags, p->long_bags + p->T);
  bool all_vec16 = true;
  for (int t = 0; t < P.T; ++t) {
    const int D = P.D[t];
    if (D < 4 || D > kMaxD || D % 4 != 0) return TBE_ERR_UNSUPPORTED;
    if (P.E[t] < 1) return TBE_ERR_INVALID_ARG;
    P.total_rows += P.E[t];
    P.total_D += D;
    if (D > P.max_D) P.max_D = D;
    if ((static_cast<int64_t>(D) * P.wbytes) % 16 != 0) all_vec16 = false;
  }
  P.vec_bytes = all_vec16 ? 16 : 8;
  if (P.itype == TBE_I32 && (P.total_rows > INT32_MAX || P.num_indices > INT32_MAX)) return TBE_ERR_RANGE;
  if (P.B >= (int64_t(1) << 31) || P.num_indices > kMaxIndices ||
      P.total_rows >= (int64_t(1) << 31))
    return TBE_ERR_UNSUPPORTED;
  return TBE_OK;
}

tbe_status device_info(DeviceInfo* out) {
  static std::mutex mu;
  static int sms_by_dev[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cuda_status(cudaGetLastError());
  out->id = dev;
  if (dev >= 0 && dev < 64) {
    std::lock_guard<std::mutex> lock(mu);
    if (sms_by_dev[dev] == 0) {
      int sms = 0;
      cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      if (e != cudaSuccess) return cuda_status(e);
      sms_by_dev[dev] = sms;
    }
    out->sms = sms_by_dev[dev];
  } else {
    int sms = 0;
    cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_status(e);
    out->sms = sms;
  }
  return TBE_OK;
}

bool hist_forward_eligible(const Problem& P, const tbe_options& o, int t) {
  return o.histogram && histogram_supported() && P.wdtype == TBE_F16 && !P.weighted &&
         P.pooling == TBE_POOL_SUM && P.E[t] <= 64 &&
         P.D[t] >= 64 && P.D[t] <= 128 && P.long_bags[t] != 0;
}

BwdLayout make_bwd_layout(const Problem& P, const tbe_options& opt, const DeviceInfo& dev) {
  BwdLayout L;
  for (int t = 0; t < P.T && L.nhist < kMaxHistTables; ++t)
    if (hist_forward_eligible(P, opt, t)) L.hist_t[L.nhist++] = t;
  const uint32_t n_cap = static_cast<uint32_t>(P.num_indices);
  L.n_cap = n_cap;
  // key range [0, total_rows]: total_rows is the sentinel of an out-of-range id
  int bits = 1;
  while ((int64_t(1) << bits) <= P.total_rows) ++bits;
  L.key_bits = bits;
  // As few passes as 10-bit digits allow, the bits shared out as evenly as they go with the
  // wider digits at the top (the top digit's highest bit is mostly the out-of-range sentinel's).
  // Digits are at least 8 bits wide.  On the stress batch (28 key bits) 9+9+10 measures the
  // same as 10+10+10; the first pass is the slow one either way (its input is in batch order,
  // so its shared-memory scatter meets the most bank conflicts).
  L.passes = (bits + kMaxRadixBits - 1) / kMaxRadixBits;
  int covered = 0;
  for (int p = 0; p < L.passes; ++p) {
    L.pass_bits[p] = std::max(8, bits / L.passes);
    covered += L.pass_bits[p];
  }
  for (int p = L.passes - 1; covered < bits; p = p == 0 ? L.passes - 1 : p - 1) {
    ++L.pass_bits[p];
    ++covered;
  }
  L.radix_bits = 8;
  for (int p = 0; p < L.passes; ++p) L.radix_bits = std::max(L.radix_bits, L.pass_bits[p]);
  L.final_buf = L.passes & 1;
  const int64_t tiles = (static_cast<int64_t>(n_cap) + kSortTile - 1) / kSortTile;
  int64_t sg = dev.sms * 2;  // two resident radix CTAs per SM (double-buffered tiles)
  if (sg > 1024) sg = 1024;
  if (tiles < sg) sg = tiles;
  L.sort_grid = static_cast<int>(sg < 1 ? 1 : sg);
  int64_t rg = dev.sms * 4;
  if (rg > 1024) rg = 1024;
  const int64_t rtiles = (static_cast<int64_t>(n_cap) + 4095) / 4096;
  if (rtiles < rg) rg = rtiles;
  L.rle_grid = static_cast<int>(rg < 1 ? 1 : rg);
  const int64_t u = std::min<int64_t>(n_cap, P.total_rows + 1);
  L.u_cap = static_cast<uint32_t>(u < 1 ? 1 : u);
  int64_t rows_in_bucket[kNumBuckets] = {0};
  for (int t = 0; t < P.T; ++t) rows_in_bucket[bucket_of(P.D[t])] += P.E[t];
  for (int k = 0; k < kNumBuckets; ++k)
    L.short_cap[k] = static_cast<uint32_t>(std::min<int64_t>(rows_in_bucket[k], n_cap));
  L.long_cap = n_cap / static_cast<uint32_t>(opt.long_threshold);
  L.chunk_cap = L.long_cap == 0 ? 0 : L.long_cap + n_cap / static_cast<uint32_t>(opt.chunk) + 1;
  L.acc_bytes = P.wdtype == TBE_F32 ? 8 : 4;
  int64_t cg = dev.sms * 4;
  if (cg > 1024) cg = 1024;
  const int64_t ctiles = (static_cast<int64_t>(L.u_cap) + 255) / 256;
  if (ctiles < cg) cg = ctiles;
  L.cls_grid = static_cast<int>(cg < 1 ? 1 : cg);

  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes, 256);
    return at;
  };
  L.counters = take(sizeof(uint32_t) * TBE_NUM_COUNTERS);
  for (int b = 0; b < 2; ++b) {
    L.keys[b] = take(sizeof(uint32_t) * n_cap);
    L.vals[b] = take(sizeof(uint32_t) * n_cap);
    L.psw[b] = P.scaled ? take(sizeof(float) * n_cap) : 0;
  }
  L.sort_counts = take(sizeof(uint32_t) * (size_t(1) << L.radix_bits) * L.sort_grid);
  L.sort_totals = take(sizeof(uint32_t) * (size_t(1) << L.radix_bits));
  L.rle_counts = take(sizeof(uint32_t) * L.rle_grid);
  L.unique = take(sizeof(uint32_t) * L.u_cap);
  L.run_off = take(sizeof(uint32_t) * (L.u_cap + 1));
  L.run_len = take(sizeof(uint32_t) * L.u_cap);
  for (int k = 0; k < kNumBuckets; ++k) L.short_list[k] = take(sizeof(uint4) * L.short_cap[k]);
  L.long_list = take(sizeof(uint32_t) * L.long_cap);
  L.chunks = take(sizeof(uint4) * L.chunk_cap);
  L.countdown = take(sizeof(uint32_t) * L.long_cap);
  L.ws_rows = take(static_cast<size_t>(L.long_cap) * P.max_D * L.acc_bytes);
  L.cls_counts = take(sizeof(uint32_t) * (kNumBuckets + 2) * L.cls_grid);
  L.hist_ws = take(kHistWsBytes * L.nhist);
  L.inv_len = P.mean_inv ? take(sizeof(float) * static_cast<size_t>(P.TB)) : 0;
  L.total = off;
  return L;
}

namespace {

BwdCtx make_ctx(const Problem& P, const tbe_options& o, const BwdLayout& L, const tbe_tables* tab,
                void* weights, float* state, const void* indices, const void* offsets,
                const float* psw, const float* grad_out, float lr, float eps, void* ws,
                int64_t* d_stats) {
  BwdCtx c;
  std::memset(&c, 0, sizeof(c));
  char* base = static_cast<char*>(ws);
  c.T = P.T;
  c.B = P.B;
  c.TB = P.TB;
  c.num_indices = P.num_indices;
  c.total_rows = P.total_rows;
  c.total_D = P.total_D;
  c.max_D = P.max_D;
  c.threshold = o.long_threshold;
  c.chunk = o.chunk;
  c.woff = tab ? tab->weight_offsets : nullptr;
  c.doff = tab ? tab->D_offsets : nullptr;
  c.roff = tab ? tab->row_offsets : nullptr;
  c.weights = weights;
  c.state = state;
  c.indices = indices;
  c.offsets = offsets;
  c.psw = psw;
  c.grad_out = grad_out;
  c.lr = lr;
  c.eps = eps;
  c.counters = reinterpret_cast<uint32_t*>(base + L.counters);
  for (int b = 0; b < 2; ++b) {
    c.keys[b] = reinterpret_cast<uint32_t*>(base + L.keys[b]);
    c.vals[b] = reinterpret_cast<uint32_t*>(base + L.vals[b]);
    c.pswbuf[b] = P.scaled ? reinterpret_cast<float*>(base + L.psw[b]) : nullptr;
  }
  c.sort_counts = reinterpret_cast<uint32_t*>(base + L.sort_counts);
  c.sort_totals = reinterpret_cast<uint32_t*>(base + L.sort_totals);
  c.rle_counts = reinterpret_cast<uint32_t*>(base + L.rle_counts);
  c.unique = reinterpret_cast<uint32_t*>(base + L.unique);
  c.run_off = reinterpret_cast<uint32_t*>(base + L.run_off);
  c.run_len = reinterpret_cast<uint32_t*>(base + L.run_len);
  for (int k = 0; k < kNumBuckets; ++k) {
    c.short_list[k] = reinterpret_cast<uint4*>(base + L.short_list[k]);
    c.short_cap[k] = L.short_cap[k];
  }
  c.long_list = reinterpret_cast<uint32_t*>(base + L.long_list);
  c.chunks = reinterpret_cast<uint4*>(base + L.chunks);
  c.countdown = reinterpret_cast<uint32_t*>(base + L.countdown);
  c.ws_rows = base + L.ws_rows;
  c.long_cap = L.long_cap;
  c.chunk_cap = L.chunk_cap;
  c.u_cap = L.u_cap;
  c.sort_grid = L.sort_grid;
  c.cls_grid = L.cls_grid;
  c.cls_counts = reinterpret_cast<uint32_t*>(base + L.cls_counts);
  c.rle_grid = L.rle_grid;
  c.stats = reinterpret_cast<unsigned long long*>(d_stats);
  c.nhist = L.nhist;
  for (int h = 0; h < kMaxHistTables; ++h) c.hist_t[h] = L.hist_t[h];
  c.hist_ws = base + L.hist_ws;
  c.inv_len = P.mean_inv ? reinterpret_cast<float*>(base + L.inv_len) : nullptr;
  return c;
}

bool tables_ok(const tbe_tables* tab) {
  return tab != nullptr && tab->weight_offsets != nullptr && tab->D_offsets != nullptr &&
         tab->row_offsets != nullptr && aligned(tab->weight_offsets, 8) && aligned(tab->D_offsets, 4) &&
         aligned(tab->row_offsets, 8);
}

// Element alignment of the buffers the kernels read or update element by element (a misaligned
// one would fault on the device instead of failing here): indices and offsets by the index
// width, fp32 arrays by 4 bytes, the int64 counters by 8 (they take 64-bit atomics).  NULL
// passes; the callers check for NULL separately.
bool elements_aligned(const Problem& P, const void* indices, const void* offsets, const float* psw,
                      const void* f32_array, const int64_t* d_stats) {
  const size_t ib = P.itype == TBE_I64 ? 8 : 4;
  return aligned(indices, ib) && aligned(offsets, ib) && aligned(psw, 4) && aligned(f32_array, 4) &&
         aligned(d_stats, 8);
}

// expand, sort, RLE and classify: the transpose half of the backward
cudaError_t run_transpose(const Problem& P, const tbe_options& o, const BwdLayout& L, const BwdCtx& c,
                          const DeviceInfo& dev, cudaStream_t s) {
  cudaError_t e;
  if ((e = cudaMemsetAsync(c.counters, 0, sizeof(uint32_t) * TBE_NUM_COUNTERS, s)) != cudaSuccess) return e;
  if ((e = launch_expand(P, c, s)) != cudaSuccess) return e;
  record(o, TBE_BWD_EV_EXPAND, s);
  if ((e = launch_sort(P, c, L, s)) != cudaSuccess) return e;
  record(o, TBE_BWD_EV_SORT, s);
  if ((e = launch_rle(P, c, L, s)) != cudaSuccess) return e;
  record(o, TBE_BWD_EV_RLE, s);
  if ((e = launch_classify(P, c, dev, o.classify_mode, s)) != cudaSuccess) return e;
  record(o, TBE_BWD_EV_CLASSIFY, s);
  return cudaSuccess;
}

}  // namespace
}  // namespace tbe

using namespace tbe;

extern "C" {

int tbe_version(void) { return TBE_VERSION; }

int tbe_last_cuda_error(void) { return g_last_cuda_error; }

const char* tbe_status_string(tbe_status status) {
  switch (status) {
    case TBE_OK: return "ok";
    case TBE_ERR_INVALID_ARG: return "invalid argument";
    case TBE_ERR_UNSUPPORTED: return "unsupported shape, dtype or size";
    case TBE_ERR_WORKSPACE: return "workspace too small";
    case TBE_ERR_CUDA: return "CUDA error";
    case TBE_ERR_RANGE: return "int32 indices requested but the range does not fit int32";
    default: return "unknown status";
  }
}

void tbe_default_options(tbe_options* opt) {
  if (opt == nullptr) return;
  std::memset(opt, 0, sizeof(*opt));
  opt->long_threshold = 256;
  opt->chunk = 256;
  opt->long_mode = TBE_LONG_AUTO;
  opt->scheduler = TBE_SCHED_PERSISTENT;
  opt->histogram = 1;
  opt->fused_bounds = 0;
  opt->events = nullptr;
  opt->num_events = 0;
  opt->launch_counter = nullptr;
  opt->classify_mode = TBE_CLASSIFY_ORDERED;
  opt->prepared = 0;
  opt->merge = TBE_MERGE_ATOMIC;
  opt->gather = TBE_GATHER_REGISTER;
}

tbe_status tbe_table_layout(const tbe_problem* prob, int64_t* weight_offsets, int32_t* D_offsets,
                            int64_t* row_offsets) {
  Problem P;
  tbe_status st = make_problem(prob, &P);
  if (st != TBE_OK) return st;
  int64_t w = 0, r = 0;
  int32_t d = 0;
  for (int t = 0; t <= P.T; ++t) {
    if (weight_offsets) weight_offsets[t] = w;
    if (D_offsets) D_offsets[t] = d;
    if (row_offsets) row_offsets[t] = r;
    if (t < P.T) {
      w += P.E[t] * P.D[t];
      d += P.D[t];
      r += P.E[t];
    }
  }
  return TBE_OK;
}

size_t tbe_bounds_workspace_size(const tbe_problem* prob) {
  Problem P;
  if (make_problem(prob, &P) != TBE_OK) return 0;
  DeviceInfo dev;
  if (device_info(&dev) != TBE_OK) return 0;
  return align_up(sizeof(int64_t) * (1 + bounds_grid(dev)), 256);
}

tbe_status tbe_bounds_check(const tbe_problem* prob, const tbe_tables* tables, void* indices,
                            void* offsets, void* ws, size_t ws_bytes, int64_t* d_stats,
                            void* stream) {
  Problem P;
  tbe_status st = make_problem(prob, &P);
  if (st != TBE_OK) return st;
  if (!tables_ok(tables) || offsets == nullptr || (P.num_indices > 0 && indices == nullptr))
    return TBE_ERR_INVALID_ARG;
  if (!elements_aligned(P, indices, offsets, nullptr, nullptr, d_stats)) return TBE_ERR_INVALID_ARG;
  DeviceInfo dev;
  if ((st = device_info(&dev)) != TBE_OK) return st;
  const int grid = bounds_grid(dev);
  if (ws == nullptr || ws_bytes < sizeof(int64_t) * (1 + grid)) return TBE_ERR_WORKSPACE;
  if (!aligned(ws, 8)) return TBE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return cuda_status(launch_bounds(P, *tables, indices, offsets, static_cast<int64_t*>(ws), grid,
                                   reinterpret_cast<unsigned long long*>(d_stats), true, s));
}

tbe_status tbe_bounds_check_offsets(const tbe_problem* prob, const tbe_tables* tables, void* offsets,
                                    void* ws, size_t ws_bytes, int64_t* d_stats, void* stream) {
  Problem P;
  tbe_status st = make_problem(prob, &P);
  if (st != TBE_OK) return st;
  if (!tables_ok(tables) || offsets == nullptr) return TBE_ERR_INVALID_ARG;
  if (!elements_aligned(P, nullptr, offsets, nullptr, nullptr, d_stats)) return TBE_ERR_INVALID_ARG;
  DeviceInfo dev;
  if ((st = device_info(&dev)) != TBE_OK) return st;
  const int grid = bounds_grid(dev);
  if (ws == nullptr || ws_bytes < sizeof(int64_t) * (1 + grid)) return TBE_ERR_WORKSPACE;
  if (!aligned(ws, 8)) return TBE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return cuda_status(launch_bounds(P, *tables, nullptr, offsets, static_cast<int64_t*>(ws), grid,
                                   reinterpret_cast<unsigned long long*>(d_stats), false, s));
}

size_t tbe_forward_workspace_size(const tbe_problem* prob, const tbe_options* opt) {
  Problem P;
  if (make_problem(prob, &P) != TBE_OK) return 0;
  const tbe_options o = resolve(opt);
  if (check_options(o) != TBE_OK) return 0;
  return static_cast<size_t>(saved_count_tables(P, o)) * static_cast<size_t>(P.B) * kHistPairsBytesPerBag;
}

tbe_status tbe_forward(const tbe_problem* prob, const tbe_options* opt, const tbe_tables* tables,
                       const void* weights, void* indices, const void* offsets, const float* psw,
                       float* out, void* ws, size_t ws_bytes, int64_t* d_stats, void* stream) {
  Problem P;
  tbe_status st = make_problem(prob, &P);
  if (st != TBE_OK) return st;
  const tbe_options o = resolve(opt);
  if ((st = check_options(o)) != TBE_OK) return st;
  if (!tables_ok(tables) || weights == nullptr || offsets == nullptr || out == nullptr ||
      (P.num_indices > 0 && indices == nullptr))
    return TBE_ERR_INVALID_ARG;
  if ((P.weighted && psw == nullptr && P.num_indices > 0) || (!P.weighted && psw != nullptr))
    return TBE_ERR_INVALID_ARG;
  if (!aligned(weights, 16) || !aligned(out, 16)) return TBE_ERR_INVALID_ARG;
  if (!elements_aligned(P, indices, offsets, psw, nullptr, d_stats)) return TBE_ERR_INVALID_ARG;
  DeviceInfo dev;
  if ((st = device_info(&dev)) != TBE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned long long* stats = reinterpret_cast<unsigned long long*>(d_stats);
  LaunchTally tally(o);
  RangeGuard ranges;
  record_fwd(o, TBE_FWD_EV_START, s);

  // Tables on the counts x table path are skipped by the gather, which walks the remaining
  // contiguous table ranges.
  std::vector<int> hist;
  for (int t = 0; t < P.T; ++t)
    if (hist_forward_eligible(P, o, t)) hist.push_back(t);
  int t0 = 0;
  size_t h = 0;
  while (t0 < P.T) {
    while (h < hist.size() && hist[h] == t0) {
      ++t0;
      ++h;
    }
    if (t0 >= P.T) break;
    int t1 = t0;
    while (t1 < P.T && !(h < hist.size() && hist[h] == t1)) ++t1;
    cudaError_t e = launch_forward_gather(P, *tables, weights, indices, offsets, psw, out, t0 * P.B,
                                          t1 * P.B, o.fused_bounds != 0, o.gather == TBE_GATHER_TMA, stats,
                                          dev, s);
    if (e == cudaSuccess)  // bags of more than a segment of lookups, summed again in segments
      e = launch_forward_long_bags(P, *tables, weights, indices, offsets, psw, out, t0 * P.B, t1 * P.B, dev, s);
    if (e != cudaSuccess) return cuda_status(e);
    t0 = t1;
  }
  record_fwd(o, TBE_FWD_EV_GATHER, s);
  // the per-bag counts of the first kMaxHistTables counts x table tables go to ws when it holds them
  const size_t saved_bytes =
      static_cast<size_t>(saved_count_tables(P, o)) * static_cast<size_t>(P.B) * kHistPairsBytesPerBag;
  uint32_t* saved = (saved_bytes > 0 && ws != nullptr && ws_bytes >= saved_bytes && aligned(ws, 16))
                        ? static_cast<uint32_t*>(ws) : nullptr;
  for (size_t h = 0; h < hist.size(); ++h) {
    const int t = hist[h];
    uint32_t* save = saved != nullptr && h < static_cast<size_t>(kMaxHistTables)
                         ? saved + h * static_cast<size_t>(P.B) * (kHistPairsBytesPerBag / 4) : nullptr;
    cudaError_t e = launch_forward_histogram(P, *tables, weights, indices, offsets, out, t, o.fused_bounds != 0,
                                             save, stats, dev, s);
    if (e == cudaSuccess)
      e = launch_forward_long_bags(P, *tables, weights, indices, offsets, psw, out, t * P.B, (t + 1) * P.B, dev, s);
    if (e != cudaSuccess) return cuda_status(e);
  }
  record_fwd(o, TBE_FWD_EV_HISTOGRAM, s);
  return TBE_OK;
}

size_t tbe_backward_workspace_size(const tbe_problem* prob, const tbe_options* opt) {
  Problem P;
  if (make_problem(prob, &P) != TBE_OK) return 0;
  const tbe_options o = resolve(opt);
  if (check_options(o) != TBE_OK) return 0;
  DeviceInfo dev;
  if (device_info(&dev) != TBE_OK) return 0;
  return make_bwd_layout(P, o, dev).total;
}

tbe_status tbe_psw_gradient(const tbe_problem* prob, const tbe_options* opt, const tbe_tables* tables,
                            const void* weights, const void* indices, const void* offsets,
                            const float* grad_out, float* grad_psw, void* stream) {
  Problem P;
  tbe_status st = make_problem(prob, &P);
  if (st != TBE_OK) return st;
  const tbe_options o = resolve(opt);
  if ((st = check_options(o)) != TBE_OK) return st;
  if (!P.weighted || !tables_ok(tables) || weights == nullptr || offsets == nullptr || grad_out == nullptr ||
      (P.num_indices > 0 && (indices == nullptr || grad_psw == nullptr)))
    return TBE_ERR_INVALID_ARG;
  if (!aligned(weights, 16) || !aligned(grad_out, 16)) return TBE_ERR_INVALID_ARG;
  if (!elements_aligned(P, indices, offsets, nullptr, grad_psw, nullptr)) return TBE_ERR_INVALID_ARG;
  DeviceInfo dev;
  if ((st = device_info(&dev)) != TBE_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  LaunchTally tally(o);
  const cudaError_t e = launch_psw_gradient(P, *tables, weights, indices, offsets, grad_out, grad_psw, dev, s);
  return e == cudaSuccess ? TBE_OK : cuda_status(e);
}

tbe_status tbe_backward_prepare(const tbe_problem* prob, const tbe_options* opt, const tbe_tables* tables,
                                const void* indices, const void* offsets, const float* psw, void* ws,
                                size_t ws_bytes, int64_t* d_stats, void* stream) {
  Problem P;
  tbe_status st = make_problem(prob, &P);
  if (st != TBE_OK) return st;
  const tbe_options o = resolve(opt);
  if ((st = check_options(o)) != TBE_OK) return st;
  if (!tables_ok(tables) || offsets == nullptr || (P.num_indices > 0 && indices == nullptr))
    return TBE_ERR_INVALID_ARG;
  if ((P.weighted && psw == nullptr && P.num_indices > 0) || (!P.weighted && psw != nullptr))
    return TBE_ERR_INVALID_ARG;
  if (!aligned(ws, 256)) return TBE_ERR_INVALID_ARG;
  if (!elements_aligned(P, indices, offsets, psw, nullptr, d_stats)) return TBE_ERR_INVALID_ARG;
  DeviceInfo dev;
  if ((st = device_info(&dev)) != TBE_OK) return st;
  const BwdLayout L = make_bwd_layout(P, o, dev);
  if (ws == nullptr || ws_bytes < L.total) return TBE_ERR_WORKSPACE;
  const BwdCtx c = make_ctx(P, o, L, tables, nullptr, nullptr, indices, offsets, psw, nullptr, 0.f, 0.f, ws,
                            d_stats);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  LaunchTally tally(o);
  RangeGuard ranges;
  record(o, TBE_BWD_EV_START, s);
  const cudaError_t e = run_transpose(P, o, L, c, dev, s);
  return e == cudaSuccess ? TBE_OK : cuda_status(e);
}

tbe_status tbe_backward_update(const tbe_problem* prob, const tbe_options* opt,
                               const tbe_tables* tables, void* weights, float* state,
                               const void* indices, const void* offsets, const float* psw,
                               const float* grad_out, tbe_optimizer optimizer, float lr, float eps,
                               void* ws, size_t ws_bytes, int64_t* d_stats, void* stream) {
  Problem P;
  tbe_status st = make_problem(prob, &P);
  if (st != TBE_OK) return st;
  const tbe_options o = resolve(opt);
  if ((st = check_options(o)) != TBE_OK) return st;
  if (optimizer != TBE_OPT_SGD && optimizer != TBE_OPT_ROWWISE_ADAGRAD) return TBE_ERR_INVALID_ARG;
  if (!tables_ok(tables) || weights == nullptr || offsets == nullptr || grad_out == nullptr ||
      (P.num_indices > 0 && indices == nullptr) ||
      (optimizer == TBE_OPT_ROWWISE_ADAGRAD && state == nullptr))
    return TBE_ERR_INVALID_ARG;
  if ((P.weighted && psw == nullptr && P.num_indices > 0) || (!P.weighted && psw != nullptr))
    return TBE_ERR_INVALID_ARG;
  if (!aligned(weights, 16) || !aligned(grad_out, 16) || !aligned(ws, 256)) return TBE_ERR_INVALID_ARG;
  if (!elements_aligned(P, indices, offsets, psw, state, d_stats)) return TBE_ERR_INVALID_ARG;
  DeviceInfo dev;
  if ((st = device_info(&dev)) != TBE_OK) return st;
  const BwdLayout L = make_bwd_layout(P, o, dev);
  if (ws == nullptr || ws_bytes < L.total) return TBE_ERR_WORKSPACE;
  const BwdCtx c = make_ctx(P, o, L, tables, weights, state, indices, offsets, psw, grad_out, lr,
                            eps, ws, d_stats);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool fused = o.long_mode != TBE_LONG_TWO_KERNEL;
  cudaError_t e;
  LaunchTally tally(o);
  RangeGuard ranges;
  record(o, TBE_BWD_EV_START, s);
  if (o.prepared) {
    // the stage events of the transpose mark the start of the update
    for (int ev : {TBE_BWD_EV_EXPAND, TBE_BWD_EV_SORT, TBE_BWD_EV_RLE, TBE_BWD_EV_CLASSIFY}) record(o, ev, s);
  } else if ((e = run_transpose(P, o, L, c, dev, s)) != cudaSuccess) {
    return cuda_status(e);
  }
  if ((e = launch_short_updates(P, c, L, optimizer, o.scheduler, dev, s)) != cudaSuccess)
    return cuda_status(e);
  record(o, TBE_BWD_EV_SHORT, s);
  if ((e = launch_long_updates(P, c, L, optimizer, fused, o.scheduler, o.merge, dev, s)) != cudaSuccess)
    return cuda_status(e);
  record(o, TBE_BWD_EV_LONG, s);
  if (!fused && (e = launch_long_apply(P, c, L, optimizer, dev, s)) != cudaSuccess) return cuda_status(e);
  record(o, TBE_BWD_EV_APPLY, s);
  if (c.nhist > 0) {
    if ((e = cudaMemsetAsync(c.hist_ws, 0, kHistWsBytes * c.nhist, s)) != cudaSuccess) return cuda_status(e);
    for (int h = 0; h < c.nhist; ++h) {
      const uint32_t* saved = o.forward_ws == nullptr ? nullptr
                              : static_cast<const uint32_t*>(o.forward_ws) +
                                    h * static_cast<size_t>(P.B) * (kHistPairsBytesPerBag / 4);
      e = launch_backward_histogram(P, c, c.hist_t[h], c.hist_ws + kHistWsBytes * h, saved, optimizer, dev, s);
      if (e != cudaSuccess) return cuda_status(e);
    }
  }
  record(o, TBE_BWD_EV_HISTOGRAM, s);
  return TBE_OK;
}

tbe_status tbe_backward_metadata(const tbe_problem* prob, const tbe_options* opt, const void* ws,
                                 size_t ws_bytes, tbe_run_metadata* meta) {
  Problem P;
  tbe_status st = make_problem(prob, &P);
  if (st != TBE_OK) return st;
  const tbe_options o = resolve(opt);
  if ((st = check_options(o)) != TBE_OK) return st;
  if (meta == nullptr || ws == nullptr) return TBE_ERR_INVALID_ARG;
  DeviceInfo dev;
  if ((st = device_info(&dev)) != TBE_OK) return st;
  const BwdLayout L = make_bwd_layout(P, o, dev);
  if (ws_bytes < L.total) return TBE_ERR_WORKSPACE;
  const char* base = static_cast<const char*>(ws);
  meta->counters = reinterpret_cast<const uint32_t*>(base + L.counters);
  meta->sorted_keys = reinterpret_cast<const uint32_t*>(base + L.keys[L.final_buf]);
  meta->sorted_bags = reinterpret_cast<const uint32_t*>(base + L.vals[L.final_buf]);
  meta->sorted_psw = P.scaled ? reinterpret_cast<const float*>(base + L.psw[L.final_buf]) : nullptr;
  meta->unique_keys = reinterpret_cast<const uint32_t*>(base + L.unique);
  meta->run_offsets = reinterpret_cast<const uint32_t*>(base + L.run_off);
  meta->run_lengths = reinterpret_cast<const uint32_t*>(base + L.run_len);
  meta->long_runs = reinterpret_cast<const uint32_t*>(base + L.long_list);
  return TBE_OK;
}

}  // extern "C"
