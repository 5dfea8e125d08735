/*
 * tbe_oracle.h -- C interface of the CPU oracle for the table-batched embedding (TBE)
 * forward and backward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  This library is the plain, slow, single-threaded reference
 * that the CUDA library is checked against.  Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark load it; the product path never does.  It shares no
 * code, header, table or helper with the CUDA library.
 *
 * Problem layout (as the pages state the problem; see each function for its source):
 *   - T tables; table t has E[t] rows of width D[t].
 *   - weights: all tables packed back to back, row-major, table t starting at element
 *     sum_{t'<t} E[t'] * D[t'].  Element type: wdtype (0 = fp32, 1 = fp16, 2 = bf16).
 *   - indices: table-local row ids, int32 (itype 0) or int64 (itype 1).
 *   - offsets: table-major bag boundaries, length T*B+1, same integer type as indices;
 *     bag (t, b) owns indices[offsets[t*B+b] .. offsets[t*B+b+1]).
 *   - psw: optional fp32 per-sample weight per index (NULL = unweighted).
 *   - pooled output / grad_output: B rows of sum_t D[t] fp32 values; table t occupies
 *     columns [sum_{t'<t} D[t'], +D[t]).
 *   - linear row id ("key") of a lookup of row i in table t: sum_{t'<t} E[t'] + i.
 *
 * Return codes: 0 = ok, -1 = invalid argument, -2 = unsupported dtype, -3 = input out of
 * range (the caller must apply oracle_bounds_repair first).
 */
#ifndef TBE_ORACLE_H
#define TBE_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

int oracle_version(void);

/* Number of short-run buckets: bucket k holds runs whose table width D has next_pow2(D) == 2^k. */
#define ORACLE_NUM_BUCKETS 11

/* Bounds/offsets repair (reading of "validates and repairs" in "Modernizing Table Batched
 * Embeddings with FBTriton", section 2, "Bounds checking"; the rule itself is not given there):
 *   offsets[T*B] is clamped into [0, num_indices]; offsets[0] := 0; every other offset is
 *   clamped into [0, offsets[T*B]] and raised to the previous (repaired) offset so that the
 *   sequence never decreases; then every index of bag (t, b) outside [0, E[t]) becomes 0.
 * Repairs are applied in place.  repaired_per_table[T] (nullable) receives the number of
 * repaired indices per table; *repaired_offsets (nullable) the number of changed offsets.
 * PARITY UNPINNED: the pages state no repair rule, so nothing outside this oracle fixes its
 * result; the tests check it only against hand-worked cases of the rule written above. */
int oracle_bounds_repair(int32_t T, int64_t B, int64_t num_indices, const int64_t* E, int32_t itype,
                         void* indices, void* offsets, int64_t* repaired_per_table,
                         int64_t* repaired_offsets);

/* Pooled forward.  pooling: 0 = sum, 1 = mean (the sum over the bag length; an empty bag
 * gives 0).  out (nullable) receives the fp32 result (round-to-nearest-even of the exact
 * value), out_exact (nullable) the fp64 value, out_absterms (nullable) the sum of |psw * w|
 * over the bag for each element (its condition scale; divided by L for mean).  All are
 * B x sum(D). */
int oracle_forward(int32_t T, int64_t B, const int32_t* D, const int64_t* E, int32_t wdtype,
                   const void* weights, int32_t itype, const void* indices, const void* offsets,
                   const float* psw, int32_t pooling, float* out, double* out_exact, double* out_absterms);

/* Backward + optimizer.  Groups the lookups by key with a std::map, sums the upstream
 * gradient rows of each key in fp64 (each scaled by its lookup's factor: psw, or 1, divided
 * by the bag length when pooling = 1 (mean)), and applies exactly one optimizer update per key:
 *   optimizer 0 (SGD):                w -= lr * g
 *   optimizer 1 (row-wise Adagrad):   s += mean_d(g_d^2);  w -= lr * g / (sqrt(s) + eps)
 * weights (wdtype) and state (fp32, one per linear row; may be NULL for SGD) are updated in
 * place with round-to-nearest-even.  Returns an opaque result handle (NULL on error, with
 * *status set) from which run metadata and exact values are read. */
void* oracle_backward(int32_t T, int64_t B, const int32_t* D, const int64_t* E, int32_t wdtype,
                      void* weights, float* state, int32_t itype, const void* indices,
                      const void* offsets, const float* psw, const float* grad_out, int32_t pooling,
                      int32_t optimizer, float lr, float eps, int32_t* status);

int64_t oracle_result_num_lookups(const void* h);  /* N = offsets[T*B] */
int64_t oracle_result_num_runs(const void* h);     /* U = number of distinct keys */
int64_t oracle_result_num_elems(const void* h);    /* sum over runs of D of the run's table */

/* Copies the result out; any pointer may be NULL.
 *   sorted_keys[N]     keys in ascending order, each repeated run-length times
 *   sorted_bags[N]     bag b of each sorted lookup; inside a run, ascending lookup position
 *   sorted_psw[N]      factor of each sorted lookup: its per-sample weight (1 when unweighted),
 *                      divided by the bag length for mean pooling, rounded to fp32
 *   unique_keys[U], run_lengths[U], run_offsets[U+1] (exclusive prefix sum, last = N)
 *   run_elem_offsets[U+1]  where run r's D values start in the three arrays below
 *   grad_sum[E]        fp64 gradient sum of each run's row
 *   w_old[E], w_exact[E]  the row before the update and the fp64 value after it
 *   state_exact[U]     fp64 optimizer state after the update (0 for SGD) */
void oracle_result_copy(const void* h, int64_t* sorted_keys, int64_t* sorted_bags, float* sorted_psw,
                        int64_t* unique_keys, int64_t* run_lengths, int64_t* run_offsets,
                        int64_t* run_elem_offsets, double* grad_sum, double* w_old,
                        double* w_exact, double* state_exact);

void oracle_result_free(void* h);

/* Gradient with respect to the per-sample weights (fp64): grad_psw[p] = sum_d
 * grad_out[b, col_t + d] * W_t[idx[p], d], divided by the bag length when pooling = 1.
 * Positions outside every bag are not written. */
int oracle_psw_gradient(int32_t T, int64_t B, const int32_t* D, const int64_t* E, int32_t wdtype,
                        const void* weights, int32_t itype, const void* indices, const void* offsets,
                        const float* grad_out, int32_t pooling, double* grad_psw);

/* Run routing ("Modernizing Table Batched Embeddings with FBTriton", section 3 and
 * section 4, Problems 1 and 3): a run is long when its length is at or above `threshold`
 * and is then split into ceil(len / chunk) chunks; a short run goes to the bucket of
 * next_pow2(D) of its table.  route[U] (nullable) receives the bucket index (log2 of
 * next_pow2(D)) of a short run or -1 for a long run. */
int oracle_classify(int32_t T, const int32_t* D, const int64_t* E, int64_t U,
                    const int64_t* unique_keys, const int64_t* run_lengths, int64_t threshold,
                    int64_t chunk, int64_t* num_short_per_bucket /* [ORACLE_NUM_BUCKETS] */,
                    int64_t* num_long, int64_t* num_chunks, int32_t* route);

/* Scalar conversions used by the oracle, exported so that the tests can check them against
 * the IEEE-754 bit layouts directly. */
double oracle_half_to_double(uint16_t h);
uint16_t oracle_double_to_half(double x);
double oracle_bf16_to_double(uint16_t h);
uint16_t oracle_double_to_bf16(double x);

#ifdef __cplusplus
}
#endif

#endif /* TBE_ORACLE_H */
