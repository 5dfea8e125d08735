// The CPU oracle built with AddressSanitizer and UndefinedBehaviorSanitizer, on small random
// problems: repair of corrupted ids and offsets, forward, backward, the gradient with respect to
// per-sample weights, routing and the 16-bit conversions.  Any invalid memory access or undefined
// behaviour aborts the program (-fno-sanitize-recover); it prints "sanitize ok" at the end.
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <random>
#include <vector>

#include "tbe_oracle.h"

namespace {

int failures = 0;
void expect(bool ok, const char* what) {
  if (!ok) {
    std::printf("FAILED: %s\n", what);
    ++failures;
  }
}

template <typename IT>
void oracle_round(std::mt19937_64& rng, int wdtype, bool weighted, int pooling, int optimizer) {
  const int T = 1 + static_cast<int>(rng() % 4);
  const int64_t B = 1 + static_cast<int64_t>(rng() % 9);
  std::vector<int32_t> D(T);
  std::vector<int64_t> E(T);
  int64_t elems = 0, rows = 0, cols = 0;
  for (int t = 0; t < T; ++t) {
    D[t] = 4 * (1 + static_cast<int>(rng() % 8));
    E[t] = 1 + static_cast<int64_t>(rng() % 50);
    elems += E[t] * D[t];
    rows += E[t];
    cols += D[t];
  }
  // bags of 0..12 lookups, then corrupted ids and offsets for the repair
  std::vector<IT> offsets(T * B + 1);
  std::vector<IT> indices;
  for (int64_t u = 0; u < T * B; ++u) {
    offsets[u] = static_cast<IT>(indices.size());
    const int t = static_cast<int>(u / B);
    const int L = static_cast<int>(rng() % 13);
    for (int k = 0; k < L; ++k) indices.push_back(static_cast<IT>(rng() % static_cast<uint64_t>(E[t])));
  }
  const int64_t N = static_cast<int64_t>(indices.size());
  offsets[T * B] = static_cast<IT>(N);
  for (auto& id : indices)
    if (rng() % 20 == 0) id = static_cast<IT>(rng() % 2 ? -1 - static_cast<int64_t>(rng() % 9) : 1000 + rng() % 9);
  for (int64_t u = 1; u < T * B; ++u)
    if (rng() % 10 == 0) offsets[u] = static_cast<IT>(static_cast<int64_t>(rng() % (N + 20)) - 10);
  std::vector<int64_t> per_table(T);
  int64_t n_off = 0;
  expect(oracle_bounds_repair(T, B, N, E.data(), sizeof(IT) == 4 ? 0 : 1, indices.data(), offsets.data(),
                              per_table.data(), &n_off) == 0,
         "bounds repair");
  const size_t wbytes = wdtype == 0 ? 4 : 2;
  std::vector<unsigned char> weights(static_cast<size_t>(elems) * wbytes);
  for (int64_t i = 0; i < elems; ++i) {
    const double x = (static_cast<double>(rng() % 2001) - 1000.0) * 1e-4;
    if (wdtype == 0) {
      const float f = static_cast<float>(x);
      std::memcpy(&weights[i * 4], &f, 4);
    } else {
      const uint16_t h = wdtype == 1 ? oracle_double_to_half(x) : oracle_double_to_bf16(x);
      std::memcpy(&weights[i * 2], &h, 2);
    }
  }
  std::vector<float> psw(N);
  for (auto& w : psw) w = static_cast<float>(rng() % 1000) * 1e-3f;
  const float* p = weighted ? psw.data() : nullptr;
  std::vector<float> out(B * cols);
  std::vector<double> exact(B * cols), absterms(B * cols);
  const int it = sizeof(IT) == 4 ? 0 : 1;
  expect(oracle_forward(T, B, D.data(), E.data(), wdtype, weights.data(), it, indices.data(), offsets.data(), p,
                        pooling, out.data(), exact.data(), absterms.data()) == 0,
         "forward");
  std::vector<float> grad(B * cols);
  for (auto& g : grad) g = (static_cast<float>(rng() % 2001) - 1000.f) * 1e-3f;
  std::vector<double> gpsw(N);
  expect(oracle_psw_gradient(T, B, D.data(), E.data(), wdtype, weights.data(), it, indices.data(), offsets.data(),
                             grad.data(), pooling, gpsw.data()) == 0,
         "psw gradient");
  std::vector<float> state(rows, 0.f);
  int32_t status = 0;
  void* h = oracle_backward(T, B, D.data(), E.data(), wdtype, weights.data(), optimizer ? state.data() : nullptr,
                            it, indices.data(), offsets.data(), p, grad.data(), pooling, optimizer, 0.01f, 1e-8f,
                            &status);
  expect(h != nullptr, "backward");
  if (h == nullptr) return;
  const int64_t n = oracle_result_num_lookups(h), U = oracle_result_num_runs(h), M = oracle_result_num_elems(h);
  std::vector<int64_t> sk(n), sb(n), uk(U), rl(U), ro(U + 1), reo(U + 1);
  std::vector<float> sp(n);
  std::vector<double> gs(M), wo(M), we(M), se(U);
  oracle_result_copy(h, sk.data(), sb.data(), sp.data(), uk.data(), rl.data(), ro.data(), reo.data(), gs.data(),
                     wo.data(), we.data(), se.data());
  oracle_result_free(h);
  int64_t total = 0;
  for (int64_t r = 0; r < U; ++r) total += rl[r];
  expect(total == n, "run lengths sum to the lookups");
  int64_t shorts[ORACLE_NUM_BUCKETS] = {0}, nl = 0, nc = 0;
  std::vector<int32_t> route(U);
  expect(oracle_classify(T, D.data(), E.data(), U, uk.data(), rl.data(), 3, 2, shorts, &nl, &nc, route.data()) == 0,
         "classify");
  // rejected arguments
  expect(oracle_forward(T, B, D.data(), E.data(), 7, weights.data(), it, indices.data(), offsets.data(), p, pooling,
                        out.data(), nullptr, nullptr) != 0,
         "bad dtype rejected");
}


}  // namespace

int main() {
  std::mt19937_64 rng(12345);
  for (uint32_t b = 0; b < 65536; ++b) {  // every 16-bit pattern through both conversions and back
    const double h = oracle_half_to_double(static_cast<uint16_t>(b));
    const double f = oracle_bf16_to_double(static_cast<uint16_t>(b));
    if (h == h) (void)oracle_double_to_half(h);
    if (f == f) (void)oracle_double_to_bf16(f);
  }
  for (int round = 0; round < 60; ++round) {
    const int wdtype = round % 3;
    const bool weighted = (round / 3) % 2 != 0;
    const int pooling = (round / 6) % 2;
    const int optimizer = (round / 12) % 2;
    if (round % 5 == 0)
      oracle_round<int32_t>(rng, wdtype, weighted, pooling, optimizer);
    else
      oracle_round<int64_t>(rng, wdtype, weighted, pooling, optimizer);
  }
  if (failures) return 1;
  std::printf("sanitize ok\n");
  return 0;
}
