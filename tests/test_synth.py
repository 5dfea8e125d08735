"""The seeded input generator: workload statistics, regeneration, and injected bad ids."""
import numpy as np
import torch

from synth import get_config, make_batch
from synth.gen import (expected_stats, grad_out_rows, grad_out_tensor, weight_rows,
                       weights_tensor, zipf_pmf, zipf_rank)


def test_large_skew_workload_hits_the_batch_statistic():
    # the pages' production batch: T*B = 4.2M bags, 83M lookups, 3M distinct rows, 125K hottest
    cfg = get_config("c3")
    assert cfg.T * cfg.B == 4_194_304
    st = expected_stats(cfg)
    assert abs(st["lookups"] / 83.9e6 - 1) < 0.01
    assert abs(st["unique"] / 3.0e6 - 1) < 0.01
    assert abs(st["hottest"] / 125e3 - 1) < 0.01


def test_zipf_sampler_matches_its_pmf():
    rng = np.random.default_rng(0)
    E, s, q = 1000, 1.3, 4.0
    k = zipf_rank(rng.random(400_000), E, s, q)
    emp = np.bincount(k, minlength=E) / k.size
    p = zipf_pmf(E, s, q)
    assert abs(p.sum() - 1) < 1e-12
    assert np.abs(emp[:20] - p[:20]).max() < 4e-3


def test_counter_values_regenerate_row_by_row():
    for name in ("c1", "c4", "c5"):
        cfg = get_config(name).shrink(B=64, E_div=1000)
        W = weights_tensor(cfg)
        rng = np.random.default_rng(1)
        for t in range(min(cfg.T, 5)):
            rows = rng.integers(0, cfg.tables[t].E, 7)
            eb = int(cfg.elem_offsets[t])
            D = cfg.tables[t].D
            full = W[eb:eb + cfg.tables[t].E * D].reshape(-1, D)[torch.from_numpy(rows)]
            assert torch.equal(full, weight_rows(cfg, t, rows))
        G = grad_out_tensor(cfg)
        bags = rng.integers(0, cfg.B, 9)
        assert torch.equal(G[torch.from_numpy(bags)], grad_out_rows(cfg, bags))
        assert abs(float(W.float().abs().max()) - cfg.w_scale) < 0.02 * cfg.w_scale + 1e-3


def test_grad_out_is_standardized():
    cfg = get_config("c2").shrink(B=512, T=4, E_div=100)
    g = grad_out_tensor(cfg).double()
    assert abs(float(g.mean())) < 0.01 and abs(float(g.var()) - 1) < 0.02


def test_batches_are_seeded_and_well_formed():
    cfg = get_config("c5").shrink(B=256, E_div=100)
    a, b = make_batch(cfg), make_batch(cfg)
    assert np.array_equal(a.indices, b.indices) and np.array_equal(a.offsets, b.offsets)
    assert a.offsets[0] == 0 and np.all(np.diff(a.offsets) >= 0) and a.offsets[-1] == a.N
    assert (np.diff(a.offsets) == 0).mean() > 0.03          # ~5% empty bags
    bad = a.bad_positions
    assert bad.size == max(1, round(a.N * cfg.bad_id_frac))
    table_of = np.searchsorted(a.offsets[::cfg.B][1:], np.arange(a.N), side="right")
    E = cfg.E[table_of]
    out_of_range = (a.indices < 0) | (a.indices >= E)
    assert np.array_equal(np.nonzero(out_of_range)[0], bad)
    assert a.psw is not None and a.psw.min() >= 0 and a.psw.max() < 1


def test_int32_workload_uses_int32():
    cfg = get_config("c2").shrink(B=128, T=3, E_div=100)
    batch = make_batch(cfg)
    assert batch.indices.dtype == np.int32 and batch.offsets.dtype == np.int32
