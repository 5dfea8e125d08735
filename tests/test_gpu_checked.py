"""The TBE_CHECKED debug flavour of the library (built from the same sources with
-DTBE_CHECKED=1): its kernels range-check the positions, run bounds and list slots they derive
from data, count each failure in TBE_STAT_CHECK_FAILED and skip the access instead of trapping.

* On valid batches it matches the oracle exactly as the default build does, with no failure.
* With the lookup count in the workspace forged lower between tbe_backward_prepare and
  tbe_backward_update, every run that ends past it fails the update kernels' range check: it is
  counted and skipped, and every other row gets its update.  (The forgery is harmless to the
  default build as well, whose arrays are sized for the true count; it is planted only into
  the checked library's workspace.)"""
import numpy as np
import pytest
import torch

from bwd_tbe_fwd_gb300 import build as tbe_build
from bwd_tbe_fwd_gb300 import tbe as T
from synth import get_config
from bwd_tbe_fwd_gb300 import TBEOptions
from tbe_harness import Case

pytestmark = pytest.mark.gpu
TBE_STAT_CHECK_FAILED = 4


@pytest.fixture(scope="module")
def checked_lib():
    path = tbe_build.build(checked=True)
    assert path.endswith("libtbe_gb300_checked.so")
    return T.load(path)


def checked_case(cfg, lib, **kw):
    case = Case(cfg, device="cuda", bounds_check=False, **kw)
    case.tbe.lib = lib
    case.run_bounds()
    return case


@pytest.mark.parametrize("name,shrink,classify", [
    ("c5", dict(B=128, T=8, E_div=500), T.TBE_CLASSIFY_ORDERED),
    ("c3", dict(B=512, T=2, E_div=2000), T.TBE_CLASSIFY_ORDERED),
    ("c3", dict(B=512, T=2, E_div=2000), T.TBE_CLASSIFY_ATOMIC),
    ("c4", dict(B=256, E_div=100), T.TBE_CLASSIFY_ORDERED),
])
def test_checked_build_matches_the_oracle_with_no_failure(checked_lib, name, shrink, classify):
    cfg = get_config(name).shrink(**shrink)
    opts = TBEOptions()
    opts.c.classify_mode = classify
    case = checked_case(cfg, checked_lib, options=opts, threshold=32, chunk=16)
    case.forward()
    case.backward()
    assert int(case.stats[TBE_STAT_CHECK_FAILED].item()) == 0


def test_checked_build_counts_and_skips_runs_past_a_corrupted_count(checked_lib):
    cfg = get_config("c3").shrink(B=512, T=2, E_div=2000)
    case = checked_case(cfg, checked_lib, threshold=32, chunk=16)
    assert case.tbe.lib is checked_lib
    tbe = case.tbe
    w0 = case.w0.to("cuda")
    grad = case.grad.to("cuda")
    state = torch.zeros(cfg.total_rows, dtype=torch.float32, device="cuda")

    def update(n_forged):
        w = w0.clone()
        s = state.clone()
        stats = torch.zeros(8, dtype=torch.int64, device="cuda")
        tbe.backward_prepare(case.idx_d, case.off_d, psw=case.psw_d, stats=stats)
        m = tbe.metadata()
        meta = (m["N"], m["unique_keys"].cpu().numpy().view(np.uint32).copy(),
                m["run_offsets"].cpu().numpy().view(np.uint32).copy())
        if n_forged is not None:
            # the classified runs stay as they are; only the lookup count the update kernels
            # check their runs against shrinks, so the runs that end past it fail the check
            m["counters_device"][T.TBE_CNT_N] = n_forged
        tbe.backward_update(w, s, case.idx_d, case.off_d, grad, psw=case.psw_d, optimizer="adagrad",
                            lr=cfg.lr, eps=cfg.eps, stats=stats, prepared=True)
        torch.cuda.synchronize()
        return w.float().cpu().numpy(), s.cpu().numpy(), stats.cpu().numpy(), meta

    w_ref, s_ref, st_ref, (N, keys, run_off) = update(None)
    n_forged = N // 2
    w_bad, s_bad, st_bad, (N2, keys2, run_off2) = update(n_forged)
    assert N2 == N and np.array_equal(keys, keys2) and np.array_equal(run_off, run_off2)
    assert st_ref[TBE_STAT_CHECK_FAILED] == 0
    past = run_off[1:] > n_forged  # runs that end past the forged count
    assert past.any() and not past.all()
    assert st_bad[TBE_STAT_CHECK_FAILED] >= int(past.sum())
    # runs that end past the forged count keep their initial row and state (a long run's chunks
    # below it are summed, but its countdown never reaches the apply); the others are updated
    # as without the forgery
    D = int(cfg.D[0])  # one width for every table of this workload: row k starts at k * D
    w0_h = w0.float().cpu().numpy()
    for r, key in enumerate(keys):
        if key >= cfg.total_rows:  # the run of out-of-range ids updates no row
            continue
        sl = slice(int(key) * D, (int(key) + 1) * D)
        if past[r]:
            assert np.array_equal(w_bad[sl], w0_h[sl]), f"run {r} past the count was applied"
            assert s_bad[key] == 0.0
        else:
            np.testing.assert_allclose(w_bad[sl], w_ref[sl], rtol=1e-3, atol=1e-6)
            np.testing.assert_allclose(s_bad[key], s_ref[key], rtol=1e-5)
