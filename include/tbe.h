/*
 * tbe.h -- C interface of the GB300 (sm_103a) table-batched embedding (TBE) library.
 *
 * What is computed (source pages by title and section):
 *   [FBT] "Modernizing Table Batched Embeddings with FBTriton"
 *   [TUT] "Table-Batched Embeddings in Triton: Gather, Pool, and Run-Length Backward"
 *
 *   Forward ([FBT] section 2; layout of [TUT] section 1): for every table t and bag b,
 *     out[b, D_offsets[t] + d] = sum over lookups p of bag (t, b) of psw[p] * W_t[indices[p], d]
 *   accumulated in fp32 (fp64 when the tables are fp32) and stored as fp32.
 *   Backward ([FBT] section 3): for every distinct (table, row) touched by the batch, the sum
 *   over its lookups of psw[p] * grad_out[b(p), D_offsets[t] + d], then exactly one SGD or
 *   row-wise Adagrad update of that row ([TUT] section 5 gives the Adagrad rule:
 *   state += mean_d(g_d^2); w -= lr * g / (sqrt(state) + eps)).
 *
 * Data layout (all device memory, caller-owned, row-major):
 *   weights        all tables packed back to back: table t starts at element
 *                  weight_offsets[t] = sum_{t'<t} E[t'] * D[t'];  row i of table t is the D[t]
 *                  contiguous elements at weight_offsets[t] + i * D[t].  fp32, fp16 or bf16.
 *   indices        [num_indices] table-local row ids, int32 or int64 (tbe_problem.itype).
 *   offsets        [T*B + 1] same integer type as indices, table-major: bag (t, b) owns
 *                  indices[offsets[t*B + b] .. offsets[t*B + b + 1]).  N = offsets[T*B].
 *   psw            [num_indices] fp32 per-sample weights (weighted problems; may be NULL when
 *                  num_indices is 0), NULL for unweighted problems.
 *   out, grad_out  [B, sum_t D[t]] fp32; table t occupies columns [D_offsets[t], +D[t]).
 *   state          [sum_t E[t]] fp32 row-wise Adagrad state, one per row, indexed by the linear
 *                  row id row_offsets[t] + i; NULL for SGD.
 *   tbe_tables     three device arrays the caller fills once with tbe_table_layout():
 *                  weight_offsets[T+1] (int64), D_offsets[T+1] (int32), row_offsets[T+1] (int64).
 *
 * Conventions:
 *   - Every call is asynchronous on `stream` (a cudaStream_t, NULL = legacy default stream).
 *     None of tbe_bounds_check, tbe_forward, tbe_backward_update synchronizes with the host,
 *     allocates memory, or copies device data to the host; every launch is sized from the
 *     host-side tbe_problem and the data-dependent counts stay on the device.
 *   - Return values report what the host can see: bad arguments, unsupported shapes, a
 *     workspace that is too small, and CUDA launch errors.  Problems found in the data
 *     (out-of-range ids, bad offsets, a bounded wait that gave up) are counted in the
 *     optional device array d_stats[TBE_NUM_STATS] (int64, accumulated; the caller zeroes it
 *     and reads it whenever it likes).  Kernels never dereference an id outside its table.
 *   - The workspace is caller-owned device memory of at least the size the matching
 *     *_workspace_size() call returns for the same problem and options; 256-byte aligned.
 *   - Limits: 1 <= T <= 4096, 0 <= B, D[t] % 4 == 0 and 4 <= D[t] <= 1024,
 *     num_indices <= 2^31 - 2^16 (lookup positions, and the few positions past a bag's end that
 *     the gather computes, stay 32-bit), sum_t E[t] < 2^31, B < 2^31; TBE_I32 additionally needs
 *     sum_t E[t] and num_indices to fit in int32 ([FBT] section 2: int32 indices/offsets when the
 *     linearized range fits below 2^31).
 */
#ifndef TBE_H
#define TBE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TBE_VERSION 1

typedef enum {
  TBE_OK = 0,
  TBE_ERR_INVALID_ARG = 1,   /* a NULL pointer, a negative size, a misaligned buffer */
  TBE_ERR_UNSUPPORTED = 2,   /* a width, dtype or size outside the limits above */
  TBE_ERR_WORKSPACE = 3,     /* ws_bytes below the size the *_workspace_size query returns */
  TBE_ERR_CUDA = 4,          /* a CUDA launch or runtime call failed */
  TBE_ERR_RANGE = 5          /* TBE_I32 requested but the rows or lookups do not fit int32 */
} tbe_status;

typedef enum { TBE_F32 = 0, TBE_F16 = 1, TBE_BF16 = 2 } tbe_dtype;
typedef enum { TBE_I32 = 0, TBE_I64 = 1 } tbe_itype;
typedef enum { TBE_POOL_SUM = 0, TBE_POOL_MEAN = 1 } tbe_pooling;
typedef enum { TBE_OPT_SGD = 0, TBE_OPT_ROWWISE_ADAGRAD = 1 } tbe_optimizer;

/* Long-run update ([FBT] section 3 and section 4, Problem 5): runs of at least
 * long_threshold lookups are split into chunks of `chunk` lookups whose partial sums meet in a
 * workspace row; the optimizer then runs either in a second kernel (TWO_KERNEL) or in the
 * same launch, by the chunk that finishes last after a device-scope fence and a countdown
 * (FUSED).  AUTO picks FUSED. */
typedef enum { TBE_LONG_AUTO = 0, TBE_LONG_TWO_KERNEL = 1, TBE_LONG_FUSED = 2 } tbe_long_mode;

/* Work distribution of the backward update kernels ([FBT] section 4, Problem 1, Solution 1.2):
 * GRID = each warp of one resident wave takes a fixed stride of the device-side run/chunk
 * lists (short runs: sixteen waves); PERSISTENT = a persistent
 * grid whose warps claim the next run or chunk from an atomic counter until none is left;
 * CLC = (long-run chunks; short runs as GRID) one CTA per 8 chunks (sized by the chunk
 * capacity), whose CTAs, when done, cancel a CTA that has not started (cluster launch control,
 * sm_100+) and process its chunks instead. */
typedef enum { TBE_SCHED_GRID = 0, TBE_SCHED_PERSISTENT = 1, TBE_SCHED_CLC = 2 } tbe_scheduler;
/* (PERSISTENT is the default: on the 83.9M-lookup stress batch it takes the short runs from 2.0
 * to 1.45 ms and the long chunks from 3.5 to 3.1 ms; CLC gives 3.3 ms for the chunks.) */

/* How a long-run chunk merges its partial sum into the run's workspace row ([FBT] section 4,
 * Problem 6): ATOMIC = vector atomic adds from registers (red.global.add.v4.f32); BULK = the
 * warp stages the row in shared memory and one lane issues a bulk reduction
 * (cp.reduce.async.bulk .add) of the whole row, performed in L2 (falls back to ATOMIC when a
 * CTA's rows would exceed 48 KB of shared memory). */
typedef enum { TBE_MERGE_ATOMIC = 0, TBE_MERGE_BULK = 1 } tbe_merge_mode;

/* How the run classifier compacts runs into its lists ([FBT] section 4, Problem 4: one reservation
 * per block per list, offsets inside the block from prefix sums, counts kept on the device):
 * ATOMIC reserves with one atomicAdd per block per list, so the lists come out in block
 * completion order; ORDERED reserves with a scan over the blocks' counts (no atomics, three
 * launches), so the lists are in key order.  Both give the same updates and counts.  ORDERED is
 * the default: with the PERSISTENT scheduler the warps then work through one table's rows at a
 * time, whose gradient slice stays in L2 (stress batch: long chunks 3.1 -> 1.9 ms, short runs
 * 1.43 -> 1.22 ms). */
typedef enum { TBE_CLASSIFY_ATOMIC = 0, TBE_CLASSIFY_ORDERED = 1 } tbe_classify_mode;

/* How the forward gather brings rows in ([FBT] section 2, "The general gather path": several
 * row loads in flight per warp).  REGISTER (the default): 16-byte row loads into registers,
 * 8 rows in flight per warp.  TMA: tables of one width D in {64, 128, 256} with 16-bit weights
 * take tile::gather4 copies of four rows of the packed [sum E, D] weights into a shared-memory
 * ring, up to 32 rows in flight per warp (other problems take REGISTER).  On the 83.9M-lookup
 * stress batch (rows mostly in L2) it measures 3.1 ms against 2.1 ms for REGISTER; on uniform
 * ids over a 1M-row table (rows from DRAM) 0.048 against 0.056 ms.  Both give the same sums. */
typedef enum { TBE_GATHER_REGISTER = 0, TBE_GATHER_TMA = 1 } tbe_gather_mode;

/* Host description of the problem.  Nothing here is read from the device. */
typedef struct {
  int32_t T;                  /* tables */
  int64_t B;                  /* bags per table (batch size) */
  int64_t num_indices;        /* length of the indices (and psw) buffers; N = offsets[T*B] <= it */
  const int32_t* D;           /* host [T] row width of each table */
  const int64_t* E;           /* host [T] rows of each table */
  tbe_dtype wdtype;           /* weight storage type; outputs and gradients are fp32 */
  tbe_itype itype;            /* type of indices AND offsets */
  int32_t weighted;           /* nonzero: per-sample weights are passed (psw must be non-NULL) */
  /* host [T] or NULL: nonzero declares that table t's bags usually hold at least 64 lookups.
   * It only steers the choice of the counts x table path ([FBT] section 2, "The small-table
   * histogram and tensor-core path"); results do not depend on it. */
  const uint8_t* long_bags;
  /* tbe_pooling: SUM, or MEAN ("Table-Batched Embeddings in Triton", "Try this": the sum
   * divided by the bag length; an empty bag gives 0).  The backward of MEAN scales each
   * lookup's gradient row by psw / L (1 / L when unweighted). */
  int32_t pooling;
} tbe_problem;

/* Device arrays describing the packed layout (see tbe_table_layout). */
typedef struct {
  const int64_t* weight_offsets;  /* [T+1] first weight element of each table */
  const int32_t* D_offsets;       /* [T+1] first output column of each table */
  const int64_t* row_offsets;     /* [T+1] first linear row of each table */
} tbe_tables;

/* Stage boundaries recorded into tbe_options.events (cudaEvent_t handles, caller-created). */
enum {
  TBE_FWD_EV_START = 0, TBE_FWD_EV_GATHER = 1, TBE_FWD_EV_HISTOGRAM = 2, TBE_FWD_NUM_EVENTS = 3
};
enum {
  TBE_BWD_EV_START = 0, TBE_BWD_EV_EXPAND = 1, TBE_BWD_EV_SORT = 2, TBE_BWD_EV_RLE = 3,
  TBE_BWD_EV_CLASSIFY = 4, TBE_BWD_EV_SHORT = 5, TBE_BWD_EV_LONG = 6, TBE_BWD_EV_APPLY = 7,
  TBE_BWD_EV_HISTOGRAM = 8, TBE_BWD_NUM_EVENTS = 9
};

typedef struct {
  int32_t long_threshold;     /* runs with at least this many lookups take the long path (256) */
  int32_t chunk;              /* lookups per long-run chunk (256) */
  int32_t long_mode;          /* tbe_long_mode */
  int32_t scheduler;          /* tbe_scheduler */
  int32_t histogram;          /* 1: use the counts x table path where eligible; 0: never */
  int32_t fused_bounds;       /* 1: tbe_forward repairs out-of-range ids in flight (writing 0 back) */
  void* const* events;        /* NULL, or cudaEvent_t[TBE_*_NUM_EVENTS] recorded at stage ends */
  int32_t num_events;
  int64_t* launch_counter;    /* NULL, or a HOST counter to which each call adds its kernel launches */
  int32_t classify_mode;      /* tbe_classify_mode */
  int32_t prepared;           /* 1: tbe_backward_update takes the transpose from ws, where
                                 tbe_backward_prepare left it, instead of computing it */
  int32_t merge;              /* tbe_merge_mode */
  int32_t gather;             /* tbe_gather_mode */
  int32_t nvtx;               /* 1: NVTX ranges (host side, one per stage: "tbe_forward.gather",
                                 "tbe_backward.sort", ...) around each stage's launches, for
                                 timeline tools; 0 (the default): none */
  const void* forward_ws;     /* Read by tbe_backward_update and tbe_backward_update_noalloc;
                                 every entry point rejects one that is not 16-byte aligned
                                 (TBE_ERR_INVALID_ARG).  NULL (the default), or the workspace
                                 of the tbe_forward call on the same batch --
                                 the same problem and options, indices and offsets, ids not
                                 changed in between -- which saved there the per-bag counts of
                                 the counts x table tables ([FBT] section 2, "Forward-state
                                 reuse"): the backward of those tables then takes their counts
                                 from it instead of reading the ids again (it still reads the ids
                                 past a bag's 256th, and does not count out-of-range ids among
                                 the first 256 a second time).  The caller answers for the
                                 match, as for `prepared`. */
} tbe_options;

/* Indices into d_stats (int64).  Counts accumulate over calls. */
enum {
  TBE_STAT_BAD_INDICES = 0,   /* out-of-range ids repaired (bounds check or fused forward) */
  TBE_STAT_BAD_OFFSETS = 1,   /* offsets changed by the offsets repair */
  TBE_STAT_UNREPAIRED = 2,    /* out-of-range ids or decreasing offsets met by a kernel that does
                                 not repair them; such lookups are skipped */
  TBE_STAT_WAIT_TIMEOUT = 3,  /* a bounded device-side wait gave up */
  TBE_STAT_CHECK_FAILED = 4,  /* a library built with TBE_CHECKED=1 found an internal index or
                                 range out of bounds (a run past the sorted lookups, a list slot
                                 past its capacity, ...) and skipped the access; always 0 in the
                                 default build, which compiles these checks out */
  TBE_NUM_STATS = 8
};

/* The defaults: threshold 256, chunk 256, AUTO long mode, PERSISTENT scheduler, histogram on,
 * fused bounds off, no events, ORDERED classifier, ATOMIC merge, REGISTER gather, no NVTX. */
void tbe_default_options(tbe_options* opt);

/* Fills the host arrays of the canonical packed layout for the problem; the caller copies
 * them to the device arrays of tbe_tables.  Any pointer may be NULL. */
tbe_status tbe_table_layout(const tbe_problem* prob, int64_t* weight_offsets /* [T+1] */,
                            int32_t* D_offsets /* [T+1] */, int64_t* row_offsets /* [T+1] */);

/* Validates and repairs indices and offsets in place ([FBT] section 2, "Bounds checking":
 * a validation step before the forward; offsets get their own small kernel).  The rule:
 * offsets[T*B] is clamped into [0, num_indices], offsets[0] becomes 0, every other offset is
 * clamped into [0, offsets[T*B]] and raised to the previous one (so bags never overlap), and
 * every id of bag (t, b) outside [0, E[t]) becomes 0.  Counts go to d_stats (nullable).
 * ws: tbe_bounds_workspace_size() bytes (may be 0 -> ws may be NULL). */
size_t tbe_bounds_workspace_size(const tbe_problem* prob);
tbe_status tbe_bounds_check(const tbe_problem* prob, const tbe_tables* tables, void* indices,
                            void* offsets, void* ws, size_t ws_bytes, int64_t* d_stats,
                            void* stream);

/* The offsets half of tbe_bounds_check alone, for callers whose tbe_forward repairs the ids in
 * flight (opt->fused_bounds = 1; [FBT] section 2: "offset validation and repair remain a
 * separate small kernel").  Same rule, workspace and counts as tbe_bounds_check. */
tbe_status tbe_bounds_check_offsets(const tbe_problem* prob, const tbe_tables* tables, void* offsets,
                                    void* ws, size_t ws_bytes, int64_t* d_stats, void* stream);

/* Pooled forward.  ws: tbe_forward_workspace_size() bytes -- 128 per bag of each counts x table
 * table (at most 8), 0 when there is none -- where the counts x table kernel saves each bag's
 * counts for a backward that reuses them (tbe_options.forward_ws); with a NULL or smaller ws
 * nothing is saved.  With opt->fused_bounds the kernels (gather and counts x table) repair
 * out-of-range ids as they read them (writing 0 back into indices, so the backward sees the
 * repaired id, counted as TBE_STAT_BAD_INDICES); without it the ids must be valid (out-of-range
 * ones are skipped and counted as TBE_STAT_UNREPAIRED).
 * Offsets must be non-decreasing (tbe_bounds_check makes them so); others are clamped so that
 * no read leaves the index array, and the bags they give are unspecified.  out: [B, sum D] fp32. */
size_t tbe_forward_workspace_size(const tbe_problem* prob, const tbe_options* opt);
tbe_status tbe_forward(const tbe_problem* prob, const tbe_options* opt, const tbe_tables* tables,
                       const void* weights, void* indices, const void* offsets, const float* psw,
                       float* out, void* ws, size_t ws_bytes, int64_t* d_stats, void* stream);

/* Backward with the optimizer applied in place: linearize the (table, row) of every lookup,
 * radix-sort the keys with their bags, run-length encode into runs, classify the runs on the
 * device (short runs bucketed by next_pow2(D), long runs split into chunks), then update each
 * touched row exactly once.  weights and state are updated in place; untouched rows are not
 * written.  lr and eps are fp32; eps is ignored for SGD. */
size_t tbe_backward_workspace_size(const tbe_problem* prob, const tbe_options* opt);
tbe_status tbe_backward_update(const tbe_problem* prob, const tbe_options* opt,
                               const tbe_tables* tables, void* weights, float* state,
                               const void* indices, const void* offsets, const float* psw,
                               const float* grad_out, tbe_optimizer optimizer, float lr, float eps,
                               void* ws, size_t ws_bytes, int64_t* d_stats, void* stream);

/* The transpose half of the backward on its own ("Modernizing Table Batched Embeddings with
 * FBTriton", section 2, "Forward-state reuse and preprocessing": the optional path that moves the
 * index transpose, sort and run-length encoding ahead of the backward): linearize, sort, run-length
 * encode and classify the batch's lookups into ws.  It reads only the layout, indices, offsets
 * and psw -- not the weights or the gradient -- so it can run before the gradient exists, e.g. on
 * a second stream alongside tbe_forward.  A later tbe_backward_update with opt->prepared = 1 and
 * the same problem, options, ws and inputs then only applies the updates.  One prepare serves one
 * update (the update consumes the long-run countdowns).  Ids must already be repaired
 * (tbe_bounds_check, or a tbe_forward with fused bounds that has finished); stats as for
 * tbe_backward_update.  The workspace size is tbe_backward_workspace_size(). */
tbe_status tbe_backward_prepare(const tbe_problem* prob, const tbe_options* opt,
                                const tbe_tables* tables, const void* indices, const void* offsets,
                                const float* psw, void* ws, size_t ws_bytes, int64_t* d_stats,
                                void* stream);

/* Gradient with respect to the per-sample weights of a weighted problem: for lookup p of bag
 * (t, b), grad_psw[p] = sum_d grad_out[b, col_t + d] * W_t[idx[p], d] (divided by the bag length
 * for MEAN pooling), accumulated in fp32 (fp64 for fp32 tables).  It reads the weights as they
 * are, so call it before tbe_backward_update changes them.  grad_psw: device fp32
 * [num_indices]; positions outside every bag are not written, lookups with an out-of-range id
 * get 0.  TBE_ERR_INVALID_ARG for an unweighted problem.  No workspace. */
tbe_status tbe_psw_gradient(const tbe_problem* prob, const tbe_options* opt, const tbe_tables* tables,
                            const void* weights, const void* indices, const void* offsets,
                            const float* grad_out, float* grad_psw, void* stream);

/* Device counters kept in the backward workspace (uint32), for the metadata view below. */
enum {
  TBE_CNT_N = 0,              /* lookups of the batch (offsets[T*B], clamped) */
  TBE_CNT_RUNS = 1,           /* U: distinct (table, row) keys */
  TBE_CNT_LONG = 2,           /* runs on the long path */
  TBE_CNT_CHUNKS = 3,         /* chunks of the long runs */
  TBE_CNT_SHORT0 = 4,         /* TBE_CNT_SHORT0 + k: short runs whose next_pow2(D) is 2^k */
  TBE_NUM_BUCKETS = 11,
  TBE_NUM_COUNTERS = 32
};

/* Where the last tbe_backward_update on this workspace left its run metadata (device
 * pointers into ws; valid until the workspace is reused).  Sizes are the device counters:
 *   sorted_keys[N], sorted_bags[N] (and sorted_psw[N] when weighted): lookups ordered by key,
 *     stable, so a run keeps its lookups in batch order; key = row_offsets[t] + row;
 *   unique_keys[U], run_offsets[U+1] (run_offsets[U] = N), run_lengths[U];
 *   long_runs[counters[TBE_CNT_LONG]]: run ids of the long runs. */
typedef struct {
  const uint32_t* counters;       /* [TBE_NUM_COUNTERS] */
  const uint32_t* sorted_keys;
  const uint32_t* sorted_bags;
  const float* sorted_psw;        /* NULL when unweighted */
  const uint32_t* unique_keys;
  const uint32_t* run_offsets;
  const uint32_t* run_lengths;
  const uint32_t* long_runs;
} tbe_run_metadata;

tbe_status tbe_backward_metadata(const tbe_problem* prob, const tbe_options* opt, const void* ws,
                                 size_t ws_bytes, tbe_run_metadata* meta);

/* Size of the scratch array built into the library for tbe_backward_update_noalloc. */
#define TBE_STATIC_SCRATCH_BYTES ((size_t)64 * 1024 * 1024)

/* tbe_backward_update for callers that cannot allocate device memory (the pages have no
 * counterpart of this entry point).  Some callers cannot hand the library a workspace: a
 * runtime whose device allocations are all planned at start-up, an allocator the calling
 * layer cannot reach, or code that must not call cudaMalloc.  This variant takes the same
 * arguments minus the workspace and uses instead a TBE_STATIC_SCRATCH_BYTES array compiled into
 * the library; it allocates nothing itself.
 *   - Limit: problems whose tbe_backward_workspace_size() exceeds TBE_STATIC_SCRATCH_BYTES are
 *     rejected with TBE_ERR_WORKSPACE; an invalid problem, options or arguments get the status
 *     tbe_backward_update would return (TBE_ERR_INVALID_ARG, TBE_ERR_UNSUPPORTED, TBE_ERR_RANGE).
 *   - Memory: the array occupies device memory from the time the library is loaded on a GPU
 *     until the process exits: with lazy module loading (CUDA's default) on every GPU where the
 *     library is used, with CUDA_MODULE_LOADING=EAGER on every GPU whose context loads the
 *     library, whether or not this entry point is called there.
 *   - Set-up: the first call on a device looks up the array's device address (with that device
 *     current) and keeps it; make that first call before any stream capture.  After a
 *     cudaDeviceReset the library must be loaded again before this entry point is used there.
 *   - Sharing: all calls on one device use the same array, which keeps the last call's
 *     contents; each call zeroes what must start at zero.  Calls whose GPU work overlaps (other
 *     streams, other host threads) race on it; the caller must order them.
 *   - opt->prepared must be 0 (TBE_ERR_INVALID_ARG otherwise): nothing prepares the array.
 * Results equal those of tbe_backward_update on the same inputs. */
tbe_status tbe_backward_update_noalloc(const tbe_problem* prob, const tbe_options* opt,
                                       const tbe_tables* tables, void* weights, float* state,
                                       const void* indices, const void* offsets, const float* psw,
                                       const float* grad_out, tbe_optimizer optimizer, float lr,
                                       float eps, int64_t* d_stats, void* stream);

const char* tbe_status_string(tbe_status status);
int tbe_version(void);
/* The cudaError_t code of the last CUDA failure reported as TBE_ERR_CUDA on this thread. */
int tbe_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* TBE_H */
