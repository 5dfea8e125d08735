"""Plants plausible mistakes in copies of the CPU oracle and checks that the pins catch each.

Every mutant below is one edit to oracle/tbe_oracle.cpp (a dropped term, a wrong sign or
index, a transposed operand, an off-by-one); the copy is compiled into a temporary directory
and must fail at least one check of tests/oracle_pins.py.  The real oracle is untouched.
"""
import os
import subprocess
import sys

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "tbe_oracle.cpp")

MUTANTS = [
    # Adagrad: sum instead of mean of g^2; eps under the root; stale state; lr dropped
    ("adagrad_sum_not_mean", "sumsq / static_cast<double>(D[t])", "sumsq"),
    ("adagrad_eps_inside_sqrt", "(std::sqrt(s_new) + static_cast<double>(eps))",
     "std::sqrt(s_new + static_cast<double>(eps))"),
    ("adagrad_state_not_updated_before_use",
     "s_new = static_cast<double>(state[key]) + sumsq", "s_new = static_cast<double>(state[key]) + 0.0 * sumsq"),
    # SGD sign
    ("sgd_sign", "w_new = w_old - static_cast<double>(lr) * r.g[d];", "w_new = w_old + static_cast<double>(lr) * r.g[d];"),
    # per-sample weights dropped in forward / backward
    ("forward_drops_psw", "const double scale = psw ? static_cast<double>(psw[p]) : 1.0;", "const double scale = 1.0;"),
    ("backward_drops_psw", "double factor = psw ? static_cast<double>(psw[p]) : 1.0;", "double factor = 1.0;"),
    # wrong gradient column (table block offset dropped) / wrong weight row base
    ("backward_grad_column", "factor * static_cast<double>(grad_out[b * width + L.col_begin[t] + d])",
     "factor * static_cast<double>(grad_out[b * width + d])"),
    ("forward_row_base", "const int64_t base = L.elem_begin[t] + row * D[t];\n        for (int32_t d = 0; d < D[t]; ++d) {\n          const double term",
     "const int64_t base = row * D[t];\n        for (int32_t d = 0; d < D[t]; ++d) {\n          const double term"),
    ("forward_output_column", "const int64_t o = b * width + L.col_begin[t] + d;", "const int64_t o = b * width + d;"),
    # grouping: payload order inside a run reversed; key without its table base
    ("run_payload_reversed", "r.bags.push_back(b);", "r.bags.insert(r.bags.begin(), b);"),
    ("key_without_table_base", "const int64_t key = L.row_begin[t] + load_int(indices, itype, p);",
     "const int64_t key = load_int(indices, itype, p) * 1 + 0 * L.row_begin[t];"),
    # routing: threshold off by one, chunk count floored, bucket off by one
    ("classify_threshold_strict", "if (run_lengths[r] >= threshold) {", "if (run_lengths[r] > threshold) {"),
    ("classify_chunks_floor", "chunks += (run_lengths[r] + chunk - 1) / chunk;", "chunks += run_lengths[r] / chunk;"),
    ("classify_bucket", "while ((1 << k) < D[t]) ++k;", "while ((1 << k) <= D[t]) ++k;"),
    # bounds: id == E accepted; offsets not made monotone
    ("bounds_accepts_E", "if (idx < 0 || idx >= E[t]) { store_int(indices, itype, p, 0); ++bad; }",
     "if (idx < 0 || idx > E[t]) { store_int(indices, itype, p, 0); ++bad; }"),
    ("bounds_no_prefix_max", "if (f < prev) f = prev;", "if (f < prev) f = f;"),
    # conversions: rounding mode (truncation) for fp16; bf16 exponent bias
    ("half_truncates", "double q = std::nearbyint(std::ldexp(a, frac_bits - e));",
     "double q = std::floor(std::ldexp(a, frac_bits - e));"),
    ("bf16_decoder_bits", "double bf16_to_double(uint16_t h) { return decode_small_float(h, 8, 7); }",
     "double bf16_to_double(uint16_t h) { return decode_small_float(h, 7, 8); }"),
    # mean pooling: divided by L + 1; backward factor without 1/L; psw gradient column / mean
    ("mean_forward_len_plus_one", "          acc[d] /= static_cast<double>(e - s);\n          absacc",
     "          acc[d] /= static_cast<double>(e - s + 1);\n          absacc"),
    ("mean_backward_unscaled", "if (pooling == 1) factor /= static_cast<double>(e - s);", "if (pooling == 1) factor /= 1.0;"),
    ("psw_grad_column", "static_cast<double>(grad_out[b * width + L.col_begin[t] + d]) * load_weight",
     "static_cast<double>(grad_out[b * width + d]) * load_weight"),
    ("psw_grad_mean_unscaled", "grad_psw[p] = pooling == 1 ? dot / static_cast<double>(e - s) : dot;", "grad_psw[p] = dot;"),
    # the forward's empty-bag/loop bound: last lookup of each bag dropped
    ("forward_drops_last_lookup",
     "for (int64_t p = s; p < e; ++p) {\n        const int64_t row = load_int(indices, itype, p);",
     "for (int64_t p = s; p + 1 < e; ++p) {\n        const int64_t row = load_int(indices, itype, p);"),
    # run metadata: run offsets not accumulated; bags numbered across tables instead of per table
    ("run_offsets_not_accumulated", "res->run_offsets.push_back(res->run_offsets.back() + len);",
     "res->run_offsets.push_back(len);"),
    ("bags_numbered_across_tables", "r.bags.push_back(b);", "r.bags.push_back(t * B + b);"),
    # Adagrad: |g| summed instead of g^2
    ("adagrad_abs_not_square", "sumsq += r.g[d] * r.g[d];", "sumsq += std::fabs(r.g[d]);"),
    # mean pooling: the empty-bag guard dropped (0 / 0)
    ("mean_empty_bag_divides", "if (pooling == 1 && e > s) {", "if (pooling == 1) {"),
    # a key on the first row of the next table attributed to the previous table
    ("table_of_key_boundary", "if (key < L.row_begin[t + 1]) return t;", "if (key <= L.row_begin[t + 1]) return t;"),
    # conversions: the fp16 overflow test off by one; the subnormal scale off by one
    ("half_overflow_boundary", "if (biased >= (1 << exp_bits) - 1) return", "if (biased > (1 << exp_bits) - 1) return"),
    ("half_subnormal_scale", "double q = std::nearbyint(std::ldexp(a, frac_bits - emin));",
     "double q = std::nearbyint(std::ldexp(a, frac_bits - emin - 1));"),
    # Adagrad: eps subtracted
    ("adagrad_eps_sign", "(std::sqrt(s_new) + static_cast<double>(eps))", "(std::sqrt(s_new) - static_cast<double>(eps))"),
    # bounds: a bad id repaired to the table's last row; the first offset left as given
    ("bounds_repairs_to_last_row", "if (idx < 0 || idx >= E[t]) { store_int(indices, itype, p, 0); ++bad; }",
     "if (idx < 0 || idx >= E[t]) { store_int(indices, itype, p, E[t] - 1); ++bad; }"),
    ("bounds_first_offset_kept", "if (TB > 0 && load_int(offsets, itype, 0) != 0) {", "if (false) {"),
]


_RUNNER = """
import sys
sys.path[:0] = [{root!r}, {tests!r}]
import oracle, oracle_pins
orc = oracle.Oracle(oracle.load({lib!r}))
failed = []
for check in oracle_pins.ALL_CHECKS:
    try:
        check(orc)
    except (AssertionError, RuntimeError) as e:
        failed.append(check.__name__)
print("FAILED:", ",".join(failed))
sys.exit(1 if failed else 0)
"""


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, old, new, tmp_path):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} must occur exactly once"
    mutated = tmp_path / "tbe_oracle.cpp"
    mutated.write_text(src.replace(old, new))
    lib_path = oracle.build(force=True, out=str(tmp_path / "liboracle_mutant.so"), src=str(mutated))
    tests_dir = os.path.dirname(os.path.abspath(__file__))
    code = _RUNNER.format(root=os.path.dirname(tests_dir), tests=tests_dir, lib=lib_path)
    # a separate process: a mutant may also crash, which counts as caught
    proc = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    assert proc.returncode != 0, f"mutant {name} passed every pin: {proc.stdout[-300:]}"
