"""CUDA library vs the CPU oracle, through the C-ABI, on the five workloads (at sizes the
oracle finishes in seconds that still span many tiles, CTAs and a ragged tail) and on the
edge cases of the method."""
import numpy as np
import pytest
import torch

import oracle
from bwd_tbe_fwd_gb300 import TBEOptions
from synth import examples, get_config
from tbe_harness import Case, check_forward, weights_to_oracle

pytestmark = pytest.mark.gpu

# Shrunk workloads: same kind (dtypes, widths, length and id laws, psw, bad ids), fewer bags,
# and rows divided so that the skew still produces runs past the 256-lookup threshold.
SMALL = {
    "c1": get_config("c1"),
    "c2": get_config("c2").shrink(B=1024, E_div=100),
    "c3": get_config("c3").shrink(B=4096, T=6, E_div=400),
    "c4": get_config("c4").shrink(B=2048, E_div=100),
    "c5": get_config("c5").shrink(B=512, E_div=100),
}


@pytest.fixture(scope="module", params=sorted(SMALL))
def case(request):
    return Case(SMALL[request.param])


def test_forward_matches_oracle(case):
    case.forward()


def test_backward_matches_oracle(case):
    res = case.backward()
    assert res["num_lookups"] > 0


def test_paths_exercised(case):
    """Every skewed workload reaches both the short and the long path."""
    m = case.tbe.metadata()
    if case.cfg.name.startswith("c1"):
        return  # uniform ids over 1000 rows: runs of length 1-2 only
    if case.counts_path_tables():
        # the skewed rows are the counts-path table's: the companion table's runs are short
        assert m["short_per_bucket"].sum() > 0 and m["N"] < case.batch.N, m["N"]
        return
    assert m["num_long"] > 0 and m["short_per_bucket"].sum() > 0, m["short_per_bucket"]


def test_bounds_repair_counts_the_injected_ids():
    cfg = SMALL["c5"]
    c = Case(cfg, bounds_check=False)
    n_bad = len(c.batch.bad_positions)
    assert n_bad > 0
    per_table, n_off = c.run_bounds()
    assert int(per_table.sum()) == n_bad and n_off == 0
    assert c.stats[0].item() == n_bad


@pytest.mark.parametrize("threshold,chunk", [(10 ** 9, 8), (8, 8), (4, 2), (1, 1), (256, 256), (64, 16)])
def test_threshold_sweep_same_answer(threshold, chunk):
    """Routing every run short, mixed, finely split or all long must not change the result."""
    c = Case(SMALL["c3"], threshold=threshold, chunk=chunk)
    c.backward()


@pytest.mark.parametrize("merge", ["atomic", "bulk"])
@pytest.mark.parametrize("long_mode", ["two_kernel", "fused"])
@pytest.mark.parametrize("scheduler", ["grid", "persistent", "clc"])
def test_long_modes_and_schedulers(long_mode, scheduler, merge):
    """Every way of distributing the long-run chunks (fixed stride, atomic claims, cluster launch
    control) and of merging their partial sums (vector atomics, bulk reductions) gives the
    oracle's updates."""
    opts = TBEOptions(long_mode={"two_kernel": 1, "fused": 2}[long_mode],
                      scheduler={"grid": 0, "persistent": 1, "clc": 2}[scheduler],
                      merge={"atomic": 0, "bulk": 1}[merge])
    for name in ("c3", "c5"):
        c = Case(SMALL[name], options=opts)
        c.backward(options=opts)


@pytest.mark.parametrize("merge", ["atomic", "bulk"])
def test_fp64_long_runs(merge):
    """fp32 tables accumulate the long runs in fp64 (an f64 bulk reduction with merge=bulk):
    every run of the tiny workload forced onto the long path in chunks of 2."""
    opts = TBEOptions(merge={"atomic": 0, "bulk": 1}[merge], scheduler=2)
    c = Case(SMALL["c1"], threshold=2, chunk=2, options=opts)
    assert c.backward(options=opts)["num_lookups"] > 0
    assert c.tbe.metadata()["num_long"] > 0


@pytest.mark.parametrize("name", ["c3", "c5", "c2"])
def test_atomic_classifier(name):
    """The pages' compaction (one atomicAdd per block per list, lists in block order) gives the
    same updates and the same route counts as the default order-preserving one."""
    opts = TBEOptions(classify_mode=0)
    c = Case(SMALL[name], options=opts)
    c.backward(options=opts)


@pytest.mark.parametrize("name", ["c3", "c5", "c2", "c1"])
def test_prepared_transpose_beside_the_forward(name):
    """tbe_backward_prepare on a second stream while the forward gather runs, then the update with
    prepared=1: the same updates and metadata as the one-call backward."""
    c = Case(SMALL[name])
    c.backward(prepared=True)


@pytest.mark.parametrize("name", ["c5", "c2", "c1", "c3"])
def test_mean_pooling(name):
    """Mean pooling ("Table-Batched Embeddings in Triton", "Try this"): the forward divides each
    bag's sum by its length (empty bags stay 0), the backward scales each lookup by psw / L (1 / L,
    taken from the offsets by the update kernels, when unweighted); the per-lookup factors the sort
    carries for weighted tables are the oracle's, bit for bit."""
    c = Case(SMALL[name], pooling="mean")
    c.forward()
    c.backward()


@pytest.mark.parametrize("pooling", ["sum", "mean"])
@pytest.mark.parametrize("name", ["c5", "c1_weighted"])
def test_psw_gradient(name, pooling):
    """Gradient with respect to the per-sample weights, against the oracle per lookup."""
    import dataclasses
    cfg = SMALL["c5"] if name == "c5" else dataclasses.replace(get_config("c1"), weighted=True, name="c1_weighted")
    c = Case(cfg, pooling=pooling)
    g = c.psw_gradient()
    assert torch.isfinite(g).all()


def test_psw_gradient_rejects_unweighted():
    from bwd_tbe_fwd_gb300.tbe import TBEError
    c = Case(SMALL["c2"])
    with pytest.raises(TBEError):
        c.tbe.psw_gradient(c.w0.cuda(), c.idx_d, c.off_d, c.grad.cuda())


def test_skewed_example_batch_routes_as_printed():
    """The tutorial's skewed batch (T=3, E=50, B=16, D=24, seed 1): the device classifier must
    produce the printed short/long/chunk counts for each threshold and chunk size."""
    import oracle_pins
    gold = oracle_pins.read_golden("skewed_batch_runs.txt")
    ex = examples.skewed_batch(seed=1)
    from bwd_tbe_fwd_gb300 import TableBatchedEmbedding
    T, E, B, D = ex["T"], ex["E"], ex["B"], ex["D"]
    grad = torch.from_numpy(examples.skewed_batch_grad(B, T * D)).cuda()
    idx = torch.from_numpy(ex["indices"]).cuda()
    off = torch.from_numpy(ex["offsets"]).cuda()
    for thr, chunk, n_short, n_long, n_chunks in gold["sweep"]:
        opts = TBEOptions(long_threshold=int(thr), chunk=int(chunk))
        tbe = TableBatchedEmbedding([D] * T, [E] * T, B, idx.numel(), torch.float32, torch.int64, options=opts)
        w = torch.from_numpy(ex["W"].reshape(-1).copy()).cuda()
        tbe.backward_update(w, None, idx, off, grad, optimizer="sgd", lr=0.05)
        torch.cuda.synchronize()
        m = tbe.metadata()
        assert m["N"] == gold["lookups"][0][0] and m["U"] == gold["unique_rows"][0][0]
        assert int(m["run_lengths"].max()) == gold["max_run"][0][0]
        assert (int(m["short_per_bucket"].sum()), m["num_long"], m["num_chunks"]) == (n_short, n_long, n_chunks)
        # and the update equals the oracle's
        w_h = ex["W"].reshape(-1).copy()
        res = oracle.backward(oracle.Tables([D] * T, [E] * T), B, w_h, None, ex["indices"], ex["offsets"],
                              grad.cpu().numpy(), optimizer="sgd", lr=0.05)
        assert np.allclose(w.cpu().numpy().astype(np.float64), w_h.astype(np.float64), rtol=1e-5, atol=1e-7)
        assert np.array_equal(m["sorted_keys"].cpu().numpy(), res["sorted_keys"])


def test_adagrad_two_steps_fp32():
    """State carried across calls (non-zero initial state) on fp32 tables with Adagrad."""
    cfg = get_config("c1").shrink(B=64, name="c1_adagrad")
    import dataclasses
    cfg = dataclasses.replace(cfg, optimizer="adagrad", lr=0.05)
    c = Case(cfg)
    c.backward(steps=2)


def test_fused_bounds_forward_repairs_in_flight():
    cfg = SMALL["c5"]
    c = Case(cfg, bounds_check=False)
    # offsets are valid in this workload; only ids are bad
    oracle.bounds_repair(c.tables, cfg.B, c.idx_h, c.off_h)
    opts = TBEOptions(fused_bounds=1)
    w_d = c.w0.cuda()
    out = c.tbe.forward(w_d, c.idx_d, c.off_d, psw=c.psw_d, stats=c.stats, options=opts)
    torch.cuda.synchronize()
    assert np.array_equal(c.idx_d.cpu().numpy(), c.idx_h)
    assert c.stats[0].item() == len(c.batch.bad_positions)
    _, exact, absterms = oracle.forward(c.tables, cfg.B, weights_to_oracle(c.w0, cfg.wdtype), c.idx_h, c.off_h,
                                        psw=c.psw_h, wdtype=cfg.wdtype)
    check_forward(out.cpu().numpy(), exact, absterms, cfg.wdtype)


def test_offsets_only_bounds_check_then_fused_forward_and_backward():
    """The split the pages describe: a small offsets kernel, ids repaired by the forward itself;
    the backward then sees the repaired ids and matches the oracle on the repaired batch."""
    cfg = SMALL["c5"]
    c = Case(cfg, bounds_check=False)
    oracle.bounds_repair(c.tables, cfg.B, c.idx_h, c.off_h)
    c.tbe.bounds_check(c.idx_d, c.off_d, stats=c.stats, offsets_only=True)
    opts = TBEOptions(fused_bounds=1)
    out = c.tbe.forward(c.w0.cuda(), c.idx_d, c.off_d, psw=c.psw_d, stats=c.stats, options=opts)
    torch.cuda.synchronize()
    assert np.array_equal(c.idx_d.cpu().numpy(), c.idx_h) and np.array_equal(c.off_d.cpu().numpy(), c.off_h)
    assert c.stats[0].item() == len(c.batch.bad_positions)
    _, exact, absterms = oracle.forward(c.tables, cfg.B, weights_to_oracle(c.w0, cfg.wdtype), c.idx_h, c.off_h,
                                        psw=c.psw_h, wdtype=cfg.wdtype)
    check_forward(out.cpu().numpy(), exact, absterms, cfg.wdtype)
    c.backward()


def corrupt_offsets(off: np.ndarray, seed: int) -> np.ndarray:
    """Offsets broken in every way the repair rule covers: a first offset that is not 0, negative
    ones, decreases, values past the last offset anywhere in the batch (clamped to N, each one
    raises every later offset to N, so the bag before the first of them takes the rest of the
    batch: hundreds of thousands of lookups of hot rows in one pooled sum), one jump far ahead
    (the prefix maximum raises every offset after it up to the jump, across the segments of many
    CTAs) and a last offset above num_indices."""
    rng = np.random.default_rng(seed)
    o = off.astype(np.int64).copy()
    TB = len(o) - 1
    N = int(o[-1])
    k = max(1, TB // 200)
    pos = rng.choice(np.arange(1, TB), size=3 * k, replace=False)
    neg, dec, past = pos[:k], pos[k:2 * k], pos[2 * k:]
    o[neg] = -rng.integers(1, 1000, size=k)
    o[dec] = o[dec] - rng.integers(1, 64, size=k)
    o[past] = N + rng.integers(1, 1000, size=k)
    o[TB // 3] = o[2 * TB // 3]
    o[0] = 7
    o[TB] = N + 50
    return o.astype(off.dtype)


@pytest.mark.parametrize("offsets_only", [False, True])
@pytest.mark.parametrize("name", ["c5", "c2"])
def test_corrupted_offsets_repaired_as_the_oracle(name, offsets_only):
    """Offsets and ids repaired on the device exactly as the oracle repairs them (bit-exact,
    with the same counts), then forward and backward parity on the repaired batch.  With
    offsets_only the ids are repaired by the forward (fused bounds) instead."""
    cfg = SMALL[name]
    c = Case(cfg, bounds_check=False)
    bad = corrupt_offsets(c.off_h, seed=17)
    c.off_h[:] = bad
    c.off_d.copy_(torch.from_numpy(bad))
    if not offsets_only:
        per_table, n_off = c.run_bounds()
        assert n_off > 0
        c.forward()
    else:
        per_table, n_off = oracle.bounds_repair(c.tables, cfg.B, c.idx_h, c.off_h)
        c.tbe.bounds_check(c.idx_d, c.off_d, stats=c.stats, offsets_only=True)
        torch.cuda.synchronize()
        assert np.array_equal(c.off_d.cpu().numpy(), c.off_h), "repaired offsets differ"
        assert c.stats[1].item() == n_off > 0
        c.forward(options=TBEOptions(fused_bounds=1))
        assert np.array_equal(c.idx_d.cpu().numpy(), c.idx_h), "ids repaired in flight differ"
        assert c.stats[0].item() == per_table.sum()
    c.backward()


def test_unrepaired_ids_are_skipped_not_dereferenced():
    cfg = SMALL["c5"]
    c = Case(cfg, bounds_check=False)
    c.tbe.forward(c.w0.cuda(), c.idx_d, c.off_d, psw=c.psw_d, stats=c.stats)
    torch.cuda.synchronize()
    n_bad = len(c.batch.bad_positions)
    assert c.stats[2].item() == n_bad
    # backward: the bad lookups form a sentinel run that is skipped
    w = c.w0.cuda()
    state = torch.zeros(cfg.total_rows, device="cuda")
    c.tbe.backward_update(w, state, c.idx_d, c.off_d, c.grad.cuda(), psw=c.psw_d, stats=c.stats)
    torch.cuda.synchronize()
    assert c.stats[2].item() == 2 * n_bad


@pytest.mark.parametrize("kind", ["all_empty", "one_bag", "single_lookup", "ragged"])
def test_edge_batches(kind):
    import dataclasses
    from synth.configs import LengthSpec
    base = get_config("c5").shrink(B=8, T=5, E_div=1000)
    if kind == "all_empty":
        tables = tuple(dataclasses.replace(t, lengths=LengthSpec("fixed", 0)) for t in base.tables)
        cfg = dataclasses.replace(base, tables=tables, bad_id_frac=0.0, name="all_empty")
    elif kind == "one_bag":
        cfg = dataclasses.replace(base.shrink(B=1, T=1), bad_id_frac=0.0, name="one_bag")
    elif kind == "single_lookup":
        tables = tuple(dataclasses.replace(t, lengths=LengthSpec("fixed", 1)) for t in base.tables[:1])
        cfg = dataclasses.replace(base, B=1, tables=tables, bad_id_frac=0.0, name="single_lookup")
    else:
        cfg = get_config("c3").shrink(B=333, T=3, E_div=4000, name="ragged")
    c = Case(cfg)
    c.forward()
    c.backward()


def test_graph_capture_no_host_sync():
    """Bounds check, forward and backward captured in one CUDA graph: capture fails on any host
    synchronization, and replays must give the eager results."""
    cfg = SMALL["c3"]
    c = Case(cfg, bounds_check=False)
    w = c.w0.cuda()
    state = torch.zeros(cfg.total_rows, device="cuda")
    grad = c.grad.cuda()
    idx0, off0 = c.idx_d.clone(), c.off_d.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # warm-up (attributes, occupancy queries) outside capture
        c.tbe.bounds_check(c.idx_d, c.off_d, stream=s)
        out = c.tbe.forward(w, c.idx_d, c.off_d, stream=s)
        c.tbe.backward_update(w, state, c.idx_d, c.off_d, grad, lr=cfg.lr, eps=cfg.eps, stream=s)
    torch.cuda.synchronize()
    w_eager, s_eager, out_eager = w.clone(), state.clone(), out.clone()
    w.copy_(c.w0.cuda())
    state.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        c.tbe.bounds_check(c.idx_d, c.off_d, stream=s)
        c.tbe.forward(w, c.idx_d, c.off_d, out=out, stream=s)
        c.tbe.backward_update(w, state, c.idx_d, c.off_d, grad, lr=cfg.lr, eps=cfg.eps, stream=s)
    w.copy_(c.w0.cuda())
    state.zero_()
    c.idx_d.copy_(idx0)
    c.off_d.copy_(off0)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, out_eager)
    # the long path merges partial sums with atomics, so only the short-run rows are bitwise
    # reproducible; compare within the fp16 tolerance
    assert torch.allclose(w.float(), w_eager.float(), rtol=2e-3, atol=1e-6)
    assert torch.allclose(state, s_eager, rtol=1e-5, atol=0)


@pytest.mark.parametrize("gather", ["register", "tma"])
@pytest.mark.parametrize("D", [100, 128, 256])
@pytest.mark.parametrize("lengths", [(600_000, 3, 7), (1_050_000,)])
def test_very_long_bags_hold_the_tolerance(lengths, D, gather):
    """Bags of 6*10^5 and 1.05*10^6 lookups of Zipf-hot fp16 rows (the stress workload's id law
    over a table of 61 rows, so the hottest rows are each added 4*10^4 - 10^5 times into one bag)
    beside short ones: every pooled element within the fp16 bound of the oracle's exact sum.  At
    D = 256 every lane of the register gather sums one column over the whole bag (at D = 128 two
    row slots share it), which is where a single fp32 running sum drifts furthest; D = 100 rows
    (200 bytes) are read as 8-byte vectors, by the register gather whichever gather is asked for."""
    import dataclasses
    from synth.configs import LengthSpec
    from bwd_tbe_fwd_gb300.tbe import TBE_GATHER_REGISTER, TBE_GATHER_TMA
    base = get_config("c3").shrink(B=len(lengths), T=1, E_div=65536, name=f"long_bags_{lengths[0]}_D{D}")
    cfg = dataclasses.replace(base, tables=tuple(dataclasses.replace(t, D=D, lengths=LengthSpec("fixed", 1))
                                                 for t in base.tables))
    c = Case(cfg, bounds_check=False)
    # bag lengths as given, ids drawn from the table's law by a second, longer draw
    big = dataclasses.replace(cfg, B=sum(lengths), name=cfg.name + "_ids")
    from synth import make_batch
    draw = make_batch(big)
    off = np.concatenate([[0], np.cumsum(lengths)]).astype(c.off_h.dtype)
    idx = draw.indices[:off[-1]].astype(c.idx_h.dtype)
    c.idx_h, c.off_h = idx.copy(), off.copy()
    c.idx_d = torch.from_numpy(idx.copy()).cuda()
    c.off_d = torch.from_numpy(off.copy()).cuda()
    c.tbe = type(c.tbe)(cfg.D, cfg.E, cfg.B, len(idx), c.tbe.weight_dtype, c.tbe.index_dtype, device="cuda")
    hot = np.bincount(idx[:lengths[0]].astype(np.int64)).max()
    assert hot > 40_000, hot
    c.forward(options=TBEOptions(gather={"register": TBE_GATHER_REGISTER, "tma": TBE_GATHER_TMA}[gather]))


def test_nvtx_ranges_option_changes_nothing():
    """With NVTX ranges on (one host-side range per stage), forward and backward give the same
    results, metadata included."""
    c = Case(SMALL["c5"], options=TBEOptions(nvtx=1))
    c.forward(options=TBEOptions(nvtx=1))
    c.backward(options=TBEOptions(nvtx=1))


def test_hundreds_of_tables():
    """300 tables of 1 to 400 rows and mixed widths (one row in some tables): gather items, the
    table search of linear keys and the per-bucket launches over many small tables."""
    import dataclasses
    import numpy as np
    from synth.configs import IdSpec, LengthSpec, TableSpec
    rng = np.random.default_rng(7)
    widths = [4, 8, 16, 24, 32, 64, 128]
    tables = tuple(TableSpec(1 if i % 50 == 0 else int(rng.integers(1, 400)), int(rng.choice(widths)),
                             LengthSpec("poisson", 3.0), IdSpec("zipf", s=1.1)) for i in range(300))
    cfg = dataclasses.replace(get_config("c5"), name="t300", B=40, tables=tables, bad_id_frac=0.0)
    c = Case(cfg, threshold=16, chunk=8)
    c.forward()
    c.backward()
