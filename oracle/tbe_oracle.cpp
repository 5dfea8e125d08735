/*
 * tbe_oracle.cpp -- plain single-threaded CPU oracle for the table-batched embedding (TBE)
 * forward pass and the backward pass with one optimizer update per touched row.
 *
 * TEST INFRASTRUCTURE ONLY: it exists so that the CUDA library can be checked against an
 * implementation that is obviously correct by reading.  It is loaded only by the tests, the
 * smoke check and the CPU-baseline leg of the benchmark.  It shares no code with the CUDA
 * library (its own packed layout, its own fp16/bf16 conversions, its own grouping), and it
 * is deliberately unblocked, unfused and unoptimised: loops in the order the method states.
 *
 * Sources (page title, section):
 *   [FBT]  "Modernizing Table Batched Embeddings with FBTriton"
 *   [TUT]  "Table-Batched Embeddings in Triton: Gather, Pool, and Run-Length Backward"
 * What each function follows is stated beside it.  Accumulation is fp64 throughout, as the
 * oracle's precision; results stored in a narrower type are rounded to nearest, ties to even.
 * Parity unpinned: oracle_bounds_repair (the pages give no repair rule; see tbe_oracle.h).
 * Every other function is pinned by the tests to values or laws outside this file.
 */
#include "tbe_oracle.h"

#include <cmath>
#include <cstdint>
#include <cstring>
#include <map>
#include <vector>

namespace {

/* ---------------------------------------------------------------------------------------
 * IEEE-754 conversions written from the bit layouts.
 *   binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 *   bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits.
 * Decoding is exact.  Encoding rounds the exact double to nearest, ties to even, directly
 * (no intermediate float, so there is no double rounding).
 * ------------------------------------------------------------------------------------- */

double decode_small_float(uint16_t bits, int exp_bits, int frac_bits) {
  const int bias = (1 << (exp_bits - 1)) - 1;
  const uint32_t sign = bits >> (exp_bits + frac_bits);
  const uint32_t e = (bits >> frac_bits) & ((1u << exp_bits) - 1);
  const uint32_t f = bits & ((1u << frac_bits) - 1);
  double mag;
  if (e == 0) {
    mag = std::ldexp(static_cast<double>(f), 1 - bias - frac_bits);  // subnormal or zero
  } else if (e == (1u << exp_bits) - 1) {
    mag = (f == 0) ? INFINITY : NAN;
  } else {
    mag = std::ldexp(static_cast<double>((1u << frac_bits) | f), static_cast<int>(e) - bias - frac_bits);
  }
  return sign ? -mag : mag;
}

uint16_t encode_small_float(double x, int exp_bits, int frac_bits) {
  const int bias = (1 << (exp_bits - 1)) - 1;
  const uint16_t exp_all_ones = static_cast<uint16_t>(((1u << exp_bits) - 1) << frac_bits);
  const uint16_t sign = std::signbit(x) ? static_cast<uint16_t>(1u << (exp_bits + frac_bits)) : 0;
  if (std::isnan(x)) return static_cast<uint16_t>(sign | exp_all_ones | (1u << (frac_bits - 1)));
  double a = std::fabs(x);
  if (std::isinf(a)) return static_cast<uint16_t>(sign | exp_all_ones);
  if (a == 0.0) return sign;
  const int emin = 1 - bias;  // exponent of the smallest normal number
  int e2;
  std::frexp(a, &e2);  // a = m * 2^e2, m in [0.5, 1)
  int e = e2 - 1;      // a = m' * 2^e, m' in [1, 2)
  if (e < emin) {
    // subnormal range: integer multiple of 2^(emin - frac_bits), rounded to nearest even
    double q = std::nearbyint(std::ldexp(a, frac_bits - emin));
    // q may round up to 2^frac_bits, which is exactly the smallest normal encoding
    return static_cast<uint16_t>(sign | static_cast<uint16_t>(q));
  }
  double q = std::nearbyint(std::ldexp(a, frac_bits - e));  // in [2^frac_bits, 2^(frac_bits+1)]
  if (q >= std::ldexp(1.0, frac_bits + 1)) {
    q = std::ldexp(q, -1);  // exact: q is 2^(frac_bits+1)
    e += 1;
  }
  const int biased = e + bias;
  if (biased >= (1 << exp_bits) - 1) return static_cast<uint16_t>(sign | exp_all_ones);  // overflow
  const uint32_t frac = static_cast<uint32_t>(q) - (1u << frac_bits);
  return static_cast<uint16_t>(sign | (static_cast<uint32_t>(biased) << frac_bits) | frac);
}

double half_to_double(uint16_t h) { return decode_small_float(h, 5, 10); }
uint16_t double_to_half(double x) { return encode_small_float(x, 5, 10); }
double bf16_to_double(uint16_t h) { return decode_small_float(h, 8, 7); }
uint16_t double_to_bf16(double x) { return encode_small_float(x, 8, 7); }

/* Element access to the weights buffer by dtype. */
double load_weight(const void* w, int32_t wdtype, int64_t i) {
  switch (wdtype) {
    case 0: return static_cast<double>(static_cast<const float*>(w)[i]);
    case 1: return half_to_double(static_cast<const uint16_t*>(w)[i]);
    default: return bf16_to_double(static_cast<const uint16_t*>(w)[i]);
  }
}

void store_weight(void* w, int32_t wdtype, int64_t i, double v) {
  switch (wdtype) {
    case 0: static_cast<float*>(w)[i] = static_cast<float>(v); break;  // C++ cast rounds to nearest even
    case 1: static_cast<uint16_t*>(w)[i] = double_to_half(v); break;
    default: static_cast<uint16_t*>(w)[i] = double_to_bf16(v); break;
  }
}

int64_t load_int(const void* p, int32_t itype, int64_t i) {
  return itype == 0 ? static_cast<int64_t>(static_cast<const int32_t*>(p)[i])
                    : static_cast<const int64_t*>(p)[i];
}

void store_int(void* p, int32_t itype, int64_t i, int64_t v) {
  if (itype == 0) static_cast<int32_t*>(p)[i] = static_cast<int32_t>(v);
  else static_cast<int64_t*>(p)[i] = v;
}

/* The packed problem layout, computed here from D and E alone ([TUT] section 1: "all tables
 * concatenated", table_off[t] = first row of table t; the output row is the concatenation
 * of the per-table pooled blocks). */
struct Layout {
  int32_t T = 0;
  std::vector<int64_t> row_begin;    // [T+1] first linear row of table t
  std::vector<int64_t> elem_begin;   // [T+1] first weight element of table t
  std::vector<int64_t> col_begin;    // [T+1] first output column of table t
};

bool make_layout(int32_t T, const int32_t* D, const int64_t* E, Layout* L) {
  if (T <= 0 || D == nullptr || E == nullptr) return false;
  L->T = T;
  L->row_begin.assign(T + 1, 0);
  L->elem_begin.assign(T + 1, 0);
  L->col_begin.assign(T + 1, 0);
  for (int32_t t = 0; t < T; ++t) {
    if (D[t] <= 0 || E[t] <= 0) return false;
    L->row_begin[t + 1] = L->row_begin[t] + E[t];
    L->elem_begin[t + 1] = L->elem_begin[t] + E[t] * static_cast<int64_t>(D[t]);
    L->col_begin[t + 1] = L->col_begin[t] + D[t];
  }
  return true;
}

int32_t table_of_key(const Layout& L, int64_t key) {
  // the table t with row_begin[t] <= key < row_begin[t+1]; plain linear scan
  for (int32_t t = 0; t < L.T; ++t)
    if (key < L.row_begin[t + 1]) return t;
  return -1;
}

/* Checks that offsets are non-decreasing within [0, num_indices] and every index lies in
 * its table; the forward and backward below assume repaired input. */
bool inputs_valid(int32_t T, int64_t B, const int64_t* E, int32_t itype, const void* indices,
                  const void* offsets) {
  const int64_t TB = static_cast<int64_t>(T) * B;
  if (load_int(offsets, itype, 0) != 0) return false;
  for (int64_t i = 0; i < TB; ++i)
    if (load_int(offsets, itype, i + 1) < load_int(offsets, itype, i)) return false;
  for (int32_t t = 0; t < T; ++t)
    for (int64_t b = 0; b < B; ++b) {
      const int64_t s = load_int(offsets, itype, t * B + b);
      const int64_t e = load_int(offsets, itype, t * B + b + 1);
      for (int64_t p = s; p < e; ++p) {
        const int64_t idx = load_int(indices, itype, p);
        if (idx < 0 || idx >= E[t]) return false;
      }
    }
  return true;
}

struct RowEntry {
  std::vector<double> g;        // fp64 gradient sum of the row
  std::vector<int64_t> bags;    // bag b of every lookup, in lookup order
  std::vector<float> psw;       // per-sample weight of every lookup
};

struct Result {
  int64_t N = 0;
  int64_t U = 0;
  int64_t elems = 0;
  std::vector<int64_t> sorted_keys, sorted_bags, unique_keys, run_lengths, run_offsets,
      run_elem_offsets;
  std::vector<float> sorted_psw;
  std::vector<double> grad_sum, w_old, w_exact, state_exact;
};

}  // namespace

extern "C" {

int oracle_version(void) { return 1; }

double oracle_half_to_double(uint16_t h) { return half_to_double(h); }
uint16_t oracle_double_to_half(double x) { return double_to_half(x); }
double oracle_bf16_to_double(uint16_t h) { return bf16_to_double(h); }
uint16_t oracle_double_to_bf16(double x) { return double_to_bf16(x); }

int oracle_bounds_repair(int32_t T, int64_t B, int64_t num_indices, const int64_t* E, int32_t itype,
                         void* indices, void* offsets, int64_t* repaired_per_table,
                         int64_t* repaired_offsets) {
  if (T <= 0 || B < 0 || num_indices < 0 || E == nullptr || offsets == nullptr) return -1;
  if (num_indices > 0 && indices == nullptr) return -1;
  if (itype != 0 && itype != 1) return -2;
  const int64_t TB = static_cast<int64_t>(T) * B;
  int64_t changed_offsets = 0;

  // 1. the last offset is the number of lookups and must lie in [0, num_indices]
  int64_t last = load_int(offsets, itype, TB);
  int64_t last_fixed = last < 0 ? 0 : (last > num_indices ? num_indices : last);
  if (last_fixed != last) { store_int(offsets, itype, TB, last_fixed); ++changed_offsets; }
  // 2. the first offset is 0 (when there is at least one bag before the last offset)
  if (TB > 0 && load_int(offsets, itype, 0) != 0) { store_int(offsets, itype, 0, 0); ++changed_offsets; }
  // 3. inner offsets: clamp into [0, last], then never below the previous offset
  int64_t prev = 0;
  for (int64_t i = 1; i < TB; ++i) {
    const int64_t o = load_int(offsets, itype, i);
    int64_t f = o < 0 ? 0 : (o > last_fixed ? last_fixed : o);
    if (f < prev) f = prev;
    if (f != o) { store_int(offsets, itype, i, f); ++changed_offsets; }
    prev = f;
  }
  // 4. indices of every bag must lie in [0, E[t]); an invalid one becomes row 0
  for (int32_t t = 0; t < T; ++t) {
    int64_t bad = 0;
    for (int64_t b = 0; b < B; ++b) {
      const int64_t s = load_int(offsets, itype, t * B + b);
      const int64_t e = load_int(offsets, itype, t * B + b + 1);
      for (int64_t p = s; p < e; ++p) {
        const int64_t idx = load_int(indices, itype, p);
        if (idx < 0 || idx >= E[t]) { store_int(indices, itype, p, 0); ++bad; }
      }
    }
    if (repaired_per_table) repaired_per_table[t] = bad;
  }
  if (repaired_offsets) *repaired_offsets = changed_offsets;
  return 0;
}

/* Forward, [FBT] section 2: for each table and bag, gather the indexed rows, optionally
 * multiply by the per-sample weight, sum, and write one D-wide pooled output; the output row
 * of sample b is [pool_t0(b) | pool_t1(b) | ...] ([TUT] section 1).  An empty bag sums to 0.
 * Mean pooling ([TUT], "Try this": divide by the bag length): the sum divided by the bag's
 * number of lookups; an empty bag gives 0, as embedding_bag(mode="mean") does. */
int oracle_forward(int32_t T, int64_t B, const int32_t* D, const int64_t* E, int32_t wdtype,
                   const void* weights, int32_t itype, const void* indices, const void* offsets,
                   const float* psw, int32_t pooling, float* out, double* out_exact, double* out_absterms) {
  Layout L;
  if (!make_layout(T, D, E, &L) || B < 0 || offsets == nullptr || weights == nullptr) return -1;
  if (wdtype < 0 || wdtype > 2 || (itype != 0 && itype != 1) || pooling < 0 || pooling > 1) return -2;
  if (!inputs_valid(T, B, E, itype, indices, offsets)) return -3;
  const int64_t width = L.col_begin[T];
  for (int64_t b = 0; b < B; ++b) {
    for (int32_t t = 0; t < T; ++t) {
      const int64_t s = load_int(offsets, itype, t * B + b);
      const int64_t e = load_int(offsets, itype, t * B + b + 1);
      std::vector<double> acc(D[t], 0.0), absacc(D[t], 0.0);
      for (int64_t p = s; p < e; ++p) {
        const int64_t row = load_int(indices, itype, p);
        const double scale = psw ? static_cast<double>(psw[p]) : 1.0;
        const int64_t base = L.elem_begin[t] + row * D[t];
        for (int32_t d = 0; d < D[t]; ++d) {
          const double term = scale * load_weight(weights, wdtype, base + d);
          acc[d] += term;
          absacc[d] += std::fabs(term);
        }
      }
      if (pooling == 1 && e > s) {
        for (int32_t d = 0; d < D[t]; ++d) {
          acc[d] /= static_cast<double>(e - s);
          absacc[d] /= static_cast<double>(e - s);
        }
      }
      for (int32_t d = 0; d < D[t]; ++d) {
        const int64_t o = b * width + L.col_begin[t] + d;
        if (out) out[o] = static_cast<float>(acc[d]);
        if (out_exact) out_exact[o] = acc[d];
        if (out_absterms) out_absterms[o] = absacc[d];
      }
    }
  }
  return 0;
}

/* Backward, [FBT] section 3: for every unique (table, row) pair touched anywhere in the
 * batch, sum the upstream gradient rows of every batch position that touched it (each
 * scaled by its per-sample weight when the table is weighted), then apply exactly one
 * optimizer update to that row.  The grouping is the transpose of [TUT] section 2:
 * linearize (table, row) into one key, order by key, one run per distinct key; inside a run
 * the lookups keep their batch order.  Here the grouping is a std::map keyed by the linear
 * row id, filled by walking the lookups in batch order.
 * Row-wise Adagrad follows [TUT] section 5: one fp32 state per row, state += mean of the
 * squared gradient over the row, then w -= lr * g / (sqrt(state) + eps). */
void* oracle_backward(int32_t T, int64_t B, const int32_t* D, const int64_t* E, int32_t wdtype,
                      void* weights, float* state, int32_t itype, const void* indices,
                      const void* offsets, const float* psw, const float* grad_out, int32_t pooling,
                      int32_t optimizer, float lr, float eps, int32_t* status) {
  int32_t dummy;
  if (!status) status = &dummy;
  Layout L;
  if (!make_layout(T, D, E, &L) || B < 0 || offsets == nullptr || weights == nullptr ||
      grad_out == nullptr || (optimizer == 1 && state == nullptr)) {
    *status = -1;
    return nullptr;
  }
  if (wdtype < 0 || wdtype > 2 || (itype != 0 && itype != 1) || optimizer < 0 || optimizer > 1 ||
      pooling < 0 || pooling > 1) {
    *status = -2;
    return nullptr;
  }
  if (!inputs_valid(T, B, E, itype, indices, offsets)) {
    *status = -3;
    return nullptr;
  }
  const int64_t width = L.col_begin[T];

  // Group: key -> (gradient sum, lookups), visiting lookups in batch (position) order.
  std::map<int64_t, RowEntry> rows;
  int64_t N = 0;
  for (int32_t t = 0; t < T; ++t) {
    for (int64_t b = 0; b < B; ++b) {
      const int64_t s = load_int(offsets, itype, t * B + b);
      const int64_t e = load_int(offsets, itype, t * B + b + 1);
      for (int64_t p = s; p < e; ++p) {
        const int64_t key = L.row_begin[t] + load_int(indices, itype, p);
        RowEntry& r = rows[key];
        if (r.g.empty()) r.g.assign(D[t], 0.0);
        // the lookup's factor: its per-sample weight, divided by the bag length when pooling by
        // mean (the derivative of the mean is the derivative of the sum over L)
        double factor = psw ? static_cast<double>(psw[p]) : 1.0;
        if (pooling == 1) factor /= static_cast<double>(e - s);
        for (int32_t d = 0; d < D[t]; ++d)
          r.g[d] += factor * static_cast<double>(grad_out[b * width + L.col_begin[t] + d]);
        r.bags.push_back(b);
        r.psw.push_back(static_cast<float>(factor));
        ++N;
      }
    }
  }
  // Table-major traversal visits positions in increasing order only if offsets are
  // table-major and non-decreasing, which inputs_valid guarantees: position p of table t
  // precedes every position of table t+1.

  Result* res = new Result();
  res->N = N;
  res->U = static_cast<int64_t>(rows.size());
  res->run_offsets.push_back(0);
  res->run_elem_offsets.push_back(0);
  for (auto& kv : rows) {
    const int64_t key = kv.first;
    RowEntry& r = kv.second;
    const int32_t t = table_of_key(L, key);
    const int64_t row = key - L.row_begin[t];
    const int64_t base = L.elem_begin[t] + row * D[t];
    const int64_t len = static_cast<int64_t>(r.bags.size());
    for (int64_t i = 0; i < len; ++i) {
      res->sorted_keys.push_back(key);
      res->sorted_bags.push_back(r.bags[i]);
      res->sorted_psw.push_back(r.psw[i]);
    }
    res->unique_keys.push_back(key);
    res->run_lengths.push_back(len);
    res->run_offsets.push_back(res->run_offsets.back() + len);
    res->run_elem_offsets.push_back(res->run_elem_offsets.back() + D[t]);

    // optimizer, in fp64 from the stored row
    double s_new = 0.0;
    if (optimizer == 1) {
      double sumsq = 0.0;
      for (int32_t d = 0; d < D[t]; ++d) sumsq += r.g[d] * r.g[d];
      s_new = static_cast<double>(state[key]) + sumsq / static_cast<double>(D[t]);
      state[key] = static_cast<float>(s_new);
    }
    for (int32_t d = 0; d < D[t]; ++d) {
      const double w_old = load_weight(weights, wdtype, base + d);
      double w_new;
      if (optimizer == 1)
        w_new = w_old - static_cast<double>(lr) * r.g[d] / (std::sqrt(s_new) + static_cast<double>(eps));
      else
        w_new = w_old - static_cast<double>(lr) * r.g[d];
      store_weight(weights, wdtype, base + d, w_new);
      res->grad_sum.push_back(r.g[d]);
      res->w_old.push_back(w_old);
      res->w_exact.push_back(w_new);
    }
    res->state_exact.push_back(s_new);
  }
  res->elems = res->run_elem_offsets.back();
  *status = 0;
  return res;
}

int64_t oracle_result_num_lookups(const void* h) { return h ? static_cast<const Result*>(h)->N : -1; }
int64_t oracle_result_num_runs(const void* h) { return h ? static_cast<const Result*>(h)->U : -1; }
int64_t oracle_result_num_elems(const void* h) { return h ? static_cast<const Result*>(h)->elems : -1; }

void oracle_result_copy(const void* h, int64_t* sorted_keys, int64_t* sorted_bags, float* sorted_psw,
                        int64_t* unique_keys, int64_t* run_lengths, int64_t* run_offsets,
                        int64_t* run_elem_offsets, double* grad_sum, double* w_old,
                        double* w_exact, double* state_exact) {
  if (!h) return;
  const Result* r = static_cast<const Result*>(h);
  auto put_i = [](int64_t* dst, const std::vector<int64_t>& v) {
    if (dst && !v.empty()) std::memcpy(dst, v.data(), v.size() * sizeof(int64_t));
  };
  auto put_d = [](double* dst, const std::vector<double>& v) {
    if (dst && !v.empty()) std::memcpy(dst, v.data(), v.size() * sizeof(double));
  };
  put_i(sorted_keys, r->sorted_keys);
  put_i(sorted_bags, r->sorted_bags);
  if (sorted_psw && !r->sorted_psw.empty())
    std::memcpy(sorted_psw, r->sorted_psw.data(), r->sorted_psw.size() * sizeof(float));
  put_i(unique_keys, r->unique_keys);
  put_i(run_lengths, r->run_lengths);
  put_i(run_offsets, r->run_offsets);
  put_i(run_elem_offsets, r->run_elem_offsets);
  put_d(grad_sum, r->grad_sum);
  put_d(w_old, r->w_old);
  put_d(w_exact, r->w_exact);
  put_d(state_exact, r->state_exact);
}

void oracle_result_free(void* h) { delete static_cast<Result*>(h); }

/* Gradient of the pooled output with respect to the per-sample weights: for lookup p of bag
 * (t, b), d out[b, cols of t] / d psw[p] = W_t[idx[p]] (divided by the bag length when pooling
 * by mean), so grad_psw[p] = sum_d grad_out[b, col_t + d] * W_t[idx[p], d] (/ L).  Computed in
 * fp64 from the weights as they are (before any update).  Positions outside every bag are
 * left untouched. */
int oracle_psw_gradient(int32_t T, int64_t B, const int32_t* D, const int64_t* E, int32_t wdtype,
                        const void* weights, int32_t itype, const void* indices, const void* offsets,
                        const float* grad_out, int32_t pooling, double* grad_psw) {
  Layout L;
  if (!make_layout(T, D, E, &L) || B < 0 || offsets == nullptr || weights == nullptr ||
      grad_out == nullptr || grad_psw == nullptr)
    return -1;
  if (wdtype < 0 || wdtype > 2 || (itype != 0 && itype != 1) || pooling < 0 || pooling > 1) return -2;
  if (!inputs_valid(T, B, E, itype, indices, offsets)) return -3;
  const int64_t width = L.col_begin[T];
  for (int32_t t = 0; t < T; ++t) {
    for (int64_t b = 0; b < B; ++b) {
      const int64_t s = load_int(offsets, itype, t * B + b);
      const int64_t e = load_int(offsets, itype, t * B + b + 1);
      for (int64_t p = s; p < e; ++p) {
        const int64_t base = L.elem_begin[t] + load_int(indices, itype, p) * D[t];
        double dot = 0.0;
        for (int32_t d = 0; d < D[t]; ++d)
          dot += static_cast<double>(grad_out[b * width + L.col_begin[t] + d]) * load_weight(weights, wdtype, base + d);
        grad_psw[p] = pooling == 1 ? dot / static_cast<double>(e - s) : dot;
      }
    }
  }
  return 0;
}

int oracle_classify(int32_t T, const int32_t* D, const int64_t* E, int64_t U,
                    const int64_t* unique_keys, const int64_t* run_lengths, int64_t threshold,
                    int64_t chunk, int64_t* num_short_per_bucket, int64_t* num_long,
                    int64_t* num_chunks, int32_t* route) {
  Layout L;
  if (!make_layout(T, D, E, &L) || U < 0 || threshold < 1 || chunk < 1) return -1;
  if (U > 0 && (unique_keys == nullptr || run_lengths == nullptr)) return -1;
  int64_t shorts[ORACLE_NUM_BUCKETS] = {0};
  int64_t longs = 0, chunks = 0;
  for (int64_t r = 0; r < U; ++r) {
    const int32_t t = table_of_key(L, unique_keys[r]);
    if (t < 0) return -3;
    if (run_lengths[r] >= threshold) {
      ++longs;
      chunks += (run_lengths[r] + chunk - 1) / chunk;
      if (route) route[r] = -1;
    } else {
      int32_t k = 0;
      while ((1 << k) < D[t]) ++k;  // 2^k = next_pow2(D)
      if (k >= ORACLE_NUM_BUCKETS) return -2;
      ++shorts[k];
      if (route) route[r] = k;
    }
  }
  if (num_short_per_bucket)
    for (int k = 0; k < ORACLE_NUM_BUCKETS; ++k) num_short_per_bucket[k] = shorts[k];
  if (num_long) *num_long = longs;
  if (num_chunks) *num_chunks = chunks;
  return 0;
}

}  // extern "C"
