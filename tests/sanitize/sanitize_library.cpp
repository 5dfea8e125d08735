// The CUDA library's host code (the problem planner, argument validation, workspace layout, the
// no-alloc entry point) built with AddressSanitizer and UndefinedBehaviorSanitizer and driven
// through its C interface on paths that return before any device work: the table layout, the
// forward workspace rule and the rejection of invalid problems, options and buffers.  Any invalid memory access or undefined
// behaviour aborts the program (-fno-sanitize-recover); it prints "sanitize ok" at the end.
#include <cstdint>
#include <cstdio>
#include <cstring>

#include "tbe.h"

namespace {

int failures = 0;
void expect(bool ok, const char* what) {
  if (!ok) {
    std::printf("FAILED: %s\n", what);
    ++failures;
  }
}

void library_validation() {
  tbe_options o;
  tbe_default_options(&o);
  const int32_t D[3] = {8, 16, 4};
  const int64_t E[3] = {10, 3, 7};
  tbe_problem p;
  std::memset(&p, 0, sizeof(p));
  p.T = 3;
  p.B = 4;
  p.num_indices = 16;
  p.D = D;
  p.E = E;
  p.wdtype = TBE_F16;
  p.itype = TBE_I64;
  int64_t woff[4], roff[4];
  int32_t doff[4];
  expect(tbe_table_layout(&p, woff, doff, roff) == TBE_OK && woff[3] == 156 && doff[3] == 28 && roff[3] == 20,
         "table layout");
  expect(tbe_table_layout(nullptr, woff, doff, roff) != TBE_OK, "layout of NULL problem rejected");
  // invalid problems
  tbe_problem q = p;
  q.T = 0;
  expect(tbe_table_layout(&q, woff, doff, roff) != TBE_OK, "T = 0 rejected");
  q = p;
  q.D = nullptr;
  expect(tbe_table_layout(&q, woff, doff, roff) != TBE_OK, "NULL widths rejected");
  const int32_t badD[3] = {8, 6, 4};
  q = p;
  q.D = badD;
  expect(tbe_table_layout(&q, woff, doff, roff) != TBE_OK, "width not a multiple of 4 rejected");
  const int64_t bigE[3] = {int64_t(1) << 30, int64_t(1) << 30, 7};
  q = p;
  q.E = bigE;
  q.itype = TBE_I32;
  expect(tbe_table_layout(&q, woff, doff, roff) != TBE_OK, "int32 rows overflow rejected");
  q = p;
  q.num_indices = -1;
  expect(tbe_bounds_workspace_size(&q) == 0, "negative lookups rejected");
  // entry points with missing buffers return before any device work
  tbe_tables tabs = {nullptr, nullptr, nullptr};
  expect(tbe_forward(&p, &o, &tabs, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, 0, nullptr, nullptr) ==
             TBE_ERR_INVALID_ARG,
         "forward without buffers rejected");
  expect(tbe_backward_update(&p, &o, &tabs, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                             TBE_OPT_ROWWISE_ADAGRAD, 0.01f, 1e-8f, nullptr, 0, nullptr, nullptr) != TBE_OK,
         "backward without buffers rejected");
  expect(tbe_bounds_check(&p, &tabs, nullptr, nullptr, nullptr, 0, nullptr, nullptr) != TBE_OK,
         "bounds check without buffers rejected");
  expect(tbe_backward_update_noalloc(&p, &o, &tabs, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                                     TBE_OPT_SGD, 0.01f, 0.f, nullptr, nullptr) != TBE_OK,
         "no-alloc backward without buffers rejected");
  tbe_options bad = o;
  bad.long_threshold = 0;
  expect(tbe_forward(&p, &bad, &tabs, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, 0, nullptr, nullptr) !=
             TBE_OK,
         "bad options rejected");
  // the forward workspace: 128 bytes per bag of each counts x table table (at most 8), none otherwise
  const int32_t hD[10] = {128, 128, 128, 128, 128, 128, 128, 128, 128, 64};
  const int64_t hE[10] = {64, 64, 64, 64, 64, 64, 64, 64, 64, 1000};
  const uint8_t hL[10] = {1, 1, 1, 1, 1, 1, 1, 1, 1, 1};
  tbe_problem h = p;
  h.T = 10;
  h.D = hD;
  h.E = hE;
  h.long_bags = hL;
  expect(tbe_forward_workspace_size(&h, &o) == size_t(8) * 4 * 128, "forward workspace: eight counts tables");
  expect(tbe_forward_workspace_size(&p, &o) == 0, "forward workspace: no counts table");
  tbe_options mis = o;
  mis.forward_ws = reinterpret_cast<const void*>(uintptr_t(4096 + 8));
  expect(tbe_forward_workspace_size(&h, &mis) == 0, "misaligned forward_ws rejected");
  expect(tbe_backward_workspace_size(&h, &mis) == 0, "misaligned forward_ws rejected by the backward");
  for (int s = 0; s <= 6; ++s) expect(tbe_status_string(static_cast<tbe_status>(s)) != nullptr, "status strings");
  expect(tbe_version() == TBE_VERSION, "version");
}

}  // namespace

int main() {
  library_validation();
  if (failures) return 1;
  std::printf("sanitize ok\n");
  return 0;
}
