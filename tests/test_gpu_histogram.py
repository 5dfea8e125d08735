"""The small-table counts x table forward and its counts^T x grad_out backward (tcgen05 tensor
cores) against the oracle and against the gather / sort paths on the same inputs."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from bwd_tbe_fwd_gb300 import TBEOptions
from synth import get_config
from synth.configs import IdSpec, LengthSpec, TableSpec
from tbe_harness import Case, check_forward, weights_to_oracle

pytestmark = pytest.mark.gpu


def hist_config(E, D, lengths, B, companion=True, bad=0.0, itype="i64", name="hist"):
    tables = [TableSpec(E, D, lengths, IdSpec("uniform"), histogram=True)]
    if companion:
        tables.append(TableSpec(5000, 64, LengthSpec("poisson", 6.0), IdSpec("uniform")))
    base = get_config("c4")
    return dataclasses.replace(base, name=name, B=B, tables=tuple(tables), bad_id_frac=bad, itype=itype)


CASES = {
    "c4_like": hist_config(64, 128, LengthSpec("fixed", 256), 2048),
    "ragged_tile_E37_D96": hist_config(37, 96, LengthSpec("poisson", 200.0), 333),
    "tail_past_256_D64": hist_config(64, 64, LengthSpec("poisson", 300.0), 200),
    "short_bags_and_empty": hist_config(50, 128, LengthSpec("poisson", 40.0, empty_frac=0.1), 130),
    "int32_ids": hist_config(64, 128, LengthSpec("fixed", 100), 256, itype="i32"),
    "alone": hist_config(64, 112, LengthSpec("fixed", 64), 1000, companion=False),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_histogram_forward_matches_oracle_and_gather(name):
    cfg = CASES[name]
    c = Case(cfg)
    out_hist = c.forward()  # default options: the histogram path serves table 0
    out_gather = c.forward(options=TBEOptions(histogram=0))
    # both within tolerance of the oracle (checked inside forward); and close to each other
    assert torch.allclose(out_hist, out_gather, rtol=1e-5, atol=1e-6)


def test_histogram_skips_out_of_range_ids():
    cfg = hist_config(64, 128, LengthSpec("fixed", 256), 512, bad=0.002, name="hist_bad")
    c = Case(cfg, bounds_check=False)
    w = c.w0.cuda()
    c.tbe.forward(w, c.idx_d, c.off_d, stats=c.stats)
    torch.cuda.synchronize()
    assert c.stats[2].item() == len(c.batch.bad_positions)
    # after repair, the histogram path equals the oracle
    c.run_bounds()
    c.forward()


@pytest.mark.parametrize("optimizer", ["adagrad", "sgd"])
@pytest.mark.parametrize("name", sorted(CASES))
def test_histogram_backward_matches_oracle(name, optimizer):
    """Table 0's update comes from counts^T x grad_out (three bf16 parts of the gradient); every
    touched row is updated once, within tolerance of the oracle; the companion table goes through
    the sort and its metadata is bit-exact."""
    c = Case(CASES[name])
    assert c.counts_path_tables() == [0]
    c.backward(optimizer=optimizer)


def test_histogram_backward_equals_sort_path():
    cfg = CASES["tail_past_256_D64"]
    c = Case(cfg)
    w_sort = c.w0.cuda()
    w_hist = c.w0.cuda()
    s_sort = torch.zeros(cfg.total_rows, device="cuda")
    s_hist = torch.zeros(cfg.total_rows, device="cuda")
    g = c.grad.cuda()
    off = TBEOptions(histogram=0)
    c.tbe.backward_update(w_sort, s_sort, c.idx_d, c.off_d, g, lr=cfg.lr, eps=cfg.eps, options=off)
    c.tbe.backward_update(w_hist, s_hist, c.idx_d, c.off_d, g, lr=cfg.lr, eps=cfg.eps)
    torch.cuda.synchronize()
    assert torch.allclose(w_hist.float(), w_sort.float(), rtol=2e-3, atol=1e-6)
    assert torch.allclose(s_hist, s_sort, rtol=1e-5, atol=0)
    # rows no lookup touched keep their bits on both paths
    touched = np.zeros(cfg.total_rows, dtype=bool)
    woff, roff = 0, 0
    w_mask = np.zeros(c.w0.numel(), dtype=bool)
    for t, spec in enumerate(cfg.tables):
        ids = c.idx_h[c.off_h[t * cfg.B]:c.off_h[(t + 1) * cfg.B]]
        rows = np.zeros(spec.E, dtype=bool)
        rows[ids] = True
        touched[roff:roff + spec.E] = rows
        w_mask[woff:woff + spec.E * spec.D] = ~np.repeat(rows, spec.D)
        woff += spec.E * spec.D
        roff += spec.E
    m = torch.from_numpy(w_mask).cuda()
    assert torch.equal(w_hist[m], c.w0.cuda()[m]) and torch.equal(w_sort[m], c.w0.cuda()[m])
    assert not bool(s_hist[torch.from_numpy(~touched).cuda()].any())


def test_histogram_forward_repairs_ids_in_flight():
    """fused_bounds on the counts x table path: out-of-range ids become row 0 (written back,
    counted), including ids past the 256th of a bag (the scalar tail)."""
    cfg = hist_config(64, 96, LengthSpec("poisson", 300.0), 300, bad=0.003, name="hist_fused")
    c = Case(cfg, bounds_check=False)
    n_bad = len(c.batch.bad_positions)
    assert n_bad > 0
    oracle.bounds_repair(c.tables, cfg.B, c.idx_h, c.off_h)
    c.tbe.bounds_check(c.idx_d, c.off_d, stats=c.stats, offsets_only=True)
    out = c.tbe.forward(c.w0.cuda(), c.idx_d, c.off_d, stats=c.stats, options=TBEOptions(fused_bounds=1))
    torch.cuda.synchronize()
    assert np.array_equal(c.idx_d.cpu().numpy(), c.idx_h)
    assert c.stats[0].item() == n_bad
    _, exact, absterms = oracle.forward(c.tables, cfg.B, weights_to_oracle(c.w0, cfg.wdtype), c.idx_h, c.off_h,
                                        wdtype=cfg.wdtype)
    check_forward(out.cpu().numpy(), exact, absterms, cfg.wdtype)


def test_histogram_backward_counts_out_of_range_ids():
    cfg = hist_config(64, 128, LengthSpec("fixed", 256), 512, bad=0.002, name="hist_bad_bwd")
    c = Case(cfg, bounds_check=False)
    n_bad = len(c.batch.bad_positions)
    assert n_bad > 0
    w = c.w0.cuda()
    state = torch.zeros(cfg.total_rows, device="cuda")
    c.tbe.backward_update(w, state, c.idx_d, c.off_d, c.grad.cuda(), stats=c.stats)
    torch.cuda.synchronize()
    assert c.stats[2].item() == n_bad
    # after repair the update equals the oracle's
    c.run_bounds()
    c.backward()


def saved_counts(c, table_index=0):
    """The per-bag counts the forward saved in its workspace for counts-path table `table_index`:
    [B, 64] uint16 (two 16-bit counts per 32-bit word, the lower id in the lower half)."""
    B = c.cfg.B
    n = B * 128
    raw = c.tbe.ws_forward[table_index * n:(table_index + 1) * n].view(torch.int16).cpu().numpy().view(np.uint16)
    return raw.reshape(B, 64)


@pytest.mark.parametrize("name", sorted(CASES))
def test_forward_saves_each_bags_counts(name):
    """[FBT] section 2, "Forward-state reuse": the counts x table forward leaves, per bag, the
    number of times each row appears among the bag's first 256 ids -- bit-exact against a count
    on the host."""
    cfg = CASES[name]
    c = Case(cfg)
    assert c.tbe.ws_forward.numel() >= cfg.B * 128
    c.tbe.ws_forward.fill_(0xAB)
    c.forward()
    got = saved_counts(c)
    E = cfg.tables[0].E
    expect = np.zeros((cfg.B, 64), dtype=np.uint16)
    for b in range(cfg.B):
        ids = c.idx_h[c.off_h[b]:c.off_h[b + 1]][:256].astype(np.int64)
        expect[b, :E] = np.bincount(ids, minlength=E)
    assert np.array_equal(got, expect)


@pytest.mark.parametrize("optimizer", ["adagrad", "sgd"])
@pytest.mark.parametrize("name", sorted(CASES))
def test_histogram_backward_reusing_forward_counts(name, optimizer):
    """The backward that takes table 0's counts from the forward of the same batch (reading no id
    among a bag's first 256) matches the oracle as the recounting one does."""
    c = Case(CASES[name])
    c.forward()
    c.backward(optimizer=optimizer, reuse_forward=True)


def test_histogram_forward_with_ids_not_16_byte_aligned():
    """Ids whose array starts 8 bytes past a 16-byte boundary take the scalar loads."""
    cfg = CASES["ragged_tile_E37_D96"]
    c = Case(cfg)
    buf = torch.empty(c.idx_d.numel() + 1, dtype=c.idx_d.dtype, device="cuda")
    ids = buf[1:]
    ids.copy_(c.idx_d)
    assert ids.data_ptr() % 16 == 8
    out = c.tbe.forward(c.w0.cuda(), ids, c.off_d)
    torch.cuda.synchronize()
    _, exact, absterms = oracle.forward(c.tables, cfg.B, weights_to_oracle(c.w0, cfg.wdtype), c.idx_h, c.off_h,
                                        wdtype=cfg.wdtype)
    check_forward(out.cpu().numpy(), exact, absterms, cfg.wdtype)


def test_histogram_backward_prepared_beside_the_forward_and_reusing_counts():
    """The transpose of the sort-path tables prepared on a second stream beside the forward, and
    the counts-path table's counts taken from that forward: the update matches the oracle and the
    sort-path metadata is bit-exact."""
    c = Case(CASES["c4_like"])
    c.backward(prepared=True, reuse_forward=True)


@pytest.mark.parametrize("reuse", [False, True], ids=["recount", "reuse"])
def test_more_than_eight_counts_tables(reuse):
    """Twelve tables qualify for the counts x table path: the forward serves all twelve on it,
    the backward the first eight (the rest go through the sort), and the forward saves the counts
    of those eight only."""
    spec = TableSpec(48, 64, LengthSpec("poisson", 90.0), IdSpec("uniform"), histogram=True)
    tables = (spec,) * 12 + (TableSpec(3000, 96, LengthSpec("poisson", 8.0), IdSpec("zipf", s=1.1)),)
    cfg = dataclasses.replace(get_config("c4"), name="hist12", B=160, tables=tables, bad_id_frac=0.0)
    c = Case(cfg)
    assert c.counts_path_tables() == list(range(8))
    assert c.tbe.ws_forward.numel() >= 8 * cfg.B * 128
    c.forward()
    c.backward(reuse_forward=reuse)
