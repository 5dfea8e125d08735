"""The two forward gathers (16-byte register loads, the default, and tile::gather4 copies into a
shared-memory ring, the option for equal-width 16-bit tables) against the oracle, each case in
both; plus the cases the tile::gather4 path meets in its own code: skipped ids (masked rows of a
stage),
per-sample weights and mean pooling, empty bags, and offsets that do not tile their span (the
per-bag walk it falls back to)."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from bwd_tbe_fwd_gb300 import TBEOptions
from bwd_tbe_fwd_gb300.tbe import TBE_GATHER_REGISTER, TBE_GATHER_TMA
from synth import get_config
from synth.configs import LengthSpec
from tbe_harness import Case, check_forward, weights_to_oracle

pytestmark = pytest.mark.gpu

MODES = {"tma": TBE_GATHER_TMA, "register": TBE_GATHER_REGISTER}


def uniform_cfg(name, B=1024, T=4, weighted=False, bad=0.0, D=None, empty=0.0):
    """Stress-shaped (Zipf ids, log-normal lengths, fp16 rows of one width), shrunk."""
    cfg = get_config("c3").shrink(B=B, T=T, E_div=400, name=name)
    tables = cfg.tables
    if D is not None:
        tables = tuple(dataclasses.replace(t, D=D) for t in tables)
    if empty:
        tables = tuple(dataclasses.replace(t, lengths=dataclasses.replace(t.lengths, empty_frac=empty))
                       for t in tables)
    return dataclasses.replace(cfg, tables=tables, weighted=weighted, bad_id_frac=bad, name=name)


def oracle_on_bags(c, bags):
    """The oracle's pooled rows of the given per-bag position ranges [(s, e)] (table-major,
    B per table), as one monotone batch holding each bag's ids in order."""
    cfg = c.cfg
    idx, off, psw = [], [0], []
    for s, e in bags:
        idx.append(c.idx_h[s:e])
        if c.psw_h is not None:
            psw.append(c.psw_h[s:e])
        off.append(off[-1] + (e - s))
    it = c.idx_h.dtype
    idx = np.concatenate(idx).astype(it) if idx else np.zeros(0, it)
    return oracle.forward(c.tables, cfg.B, weights_to_oracle(c.w0, cfg.wdtype), idx, np.array(off, it),
                          psw=np.concatenate(psw) if psw else None, wdtype=cfg.wdtype, pooling=c.pooling)


def run_forward(c, mode, **opts):
    out = c.tbe.forward(c.w0.cuda(), c.idx_d, c.off_d, psw=c.psw_d, stats=c.stats,
                        options=TBEOptions(gather=MODES[mode], **opts))
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("name", ["c2", "c3", "c4"])
@pytest.mark.parametrize("mode", sorted(MODES))
def test_gather_modes_match_oracle(name, mode):
    from test_gpu_parity import SMALL
    c = Case(SMALL[name])
    c.forward(options=TBEOptions(gather=MODES[mode]))


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("weighted,pooling", [(False, "sum"), (True, "sum"), (False, "mean"), (True, "mean")])
def test_tma_gather_widths_weights_pooling(D, weighted, pooling):
    c = Case(uniform_cfg(f"tma_D{D}", B=700, D=D, weighted=weighted, empty=0.05), pooling=pooling)
    for mode in MODES:
        c.forward(options=TBEOptions(gather=MODES[mode]))


def test_tma_gather_skips_unrepaired_ids():
    c = Case(uniform_cfg("tma_bad", bad=0.01), bounds_check=False)
    n_bad = len(c.batch.bad_positions)
    assert n_bad > 0
    cfg = c.cfg
    E = np.asarray(cfg.E)
    off = c.off_h.astype(np.int64)
    ok = np.ones(len(c.idx_h), dtype=bool)
    for t in range(cfg.T):
        s, e = off[t * cfg.B], off[(t + 1) * cfg.B]
        ids = c.idx_h[s:e].astype(np.int64)
        ok[s:e] = (ids >= 0) & (ids < E[t])
    # expected: the oracle on the batch without the skipped lookups
    keep = np.flatnonzero(ok)
    new_off = np.searchsorted(keep, off).astype(c.off_h.dtype)
    it = c.idx_h.dtype
    _, exact, absterms = oracle.forward(c.tables, cfg.B, weights_to_oracle(c.w0, cfg.wdtype),
                                        c.idx_h[keep].astype(it), new_off,
                                        psw=None if c.psw_h is None else c.psw_h[keep], wdtype=cfg.wdtype)
    for k, mode in enumerate(MODES):
        x = run_forward(c, mode)
        check_forward(x, exact, absterms, cfg.wdtype)
        assert c.stats[2].item() == (k + 1) * n_bad  # each skipped id counted once per forward


def test_tma_gather_repairs_ids_in_flight():
    c = Case(uniform_cfg("tma_fused", bad=0.01), bounds_check=False)
    oracle.bounds_repair(c.tables, c.cfg.B, c.idx_h, c.off_h)
    x = run_forward(c, "tma", fused_bounds=1)
    assert np.array_equal(c.idx_d.cpu().numpy(), c.idx_h), "ids repaired in flight differ from the oracle's repair"
    assert c.stats[0].item() == len(c.batch.bad_positions)
    _, exact, absterms = oracle.forward(c.tables, c.cfg.B, weights_to_oracle(c.w0, c.cfg.wdtype), c.idx_h, c.off_h,
                                        wdtype=c.cfg.wdtype)
    check_forward(x, exact, absterms, c.cfg.wdtype)


def test_untiled_offsets_take_the_per_bag_walk():
    """Offsets left unrepaired with decreases and overlaps: each bag reads its own clamped range
    [clamp(o[u], 0, N), clamp(o[u+1], that, N)) in both gathers."""
    c = Case(uniform_cfg("tma_untiled", B=512), bounds_check=False)
    rng = np.random.default_rng(21)
    off = c.off_h.astype(np.int64).copy()
    N = len(c.idx_h)
    for u in rng.choice(np.arange(1, len(off) - 1), size=40, replace=False):
        off[u] = min(N, off[u + 1] + int(rng.integers(1, 9)))  # bag u-1 runs past bag u's start
    c.off_h = off.astype(c.off_h.dtype)
    c.off_d = torch.from_numpy(c.off_h.copy()).cuda()
    bags = []
    for u in range(len(off) - 1):
        s = min(max(off[u], 0), N)
        e = min(max(off[u + 1], s), N)
        bags.append((s, e))
    _, exact, absterms = oracle_on_bags(c, bags)
    for mode in MODES:
        check_forward(run_forward(c, mode), exact, absterms, c.cfg.wdtype)


def test_tma_gather_all_empty_and_single_lookup_bags():
    for name, L in (("tma_empty", LengthSpec("fixed", 0)), ("tma_single", LengthSpec("fixed", 1))):
        cfg = uniform_cfg(name, B=300)
        cfg = dataclasses.replace(cfg, tables=tuple(dataclasses.replace(t, lengths=L) for t in cfg.tables))
        c = Case(cfg)
        for mode in MODES:
            c.forward(options=TBEOptions(gather=MODES[mode]))
