"""The CUDA library at the workloads' full sizes, in the launch configuration the benchmark times
(offsets-only bounds check with ids repaired inside the forward, default scheduler and run
lists): the large-skew batch (32 tables of 4M fp16 rows x 128, ~83.9M Zipf-skewed lookups),
the mixed batch (64 tables of widths 32-256, bf16, per-sample weights, 0.1% out-of-range ids,
~29.9M lookups), the histogram batch (a 64-row table on the counts x table path beside a 1M-row
table) and the mid batch (int32).  Each is checked against the oracle where it can follow one
output at a time and against properties that hold at any size:

  * repaired ids and offsets: bit-exact over the whole batch (the oracle's repair);
  * sorted keys, sorted bags, unique keys, run offsets and run lengths: bit-exact over the
    whole batch, against a stable host sort of the linear keys (lookups of counts-path tables
    left out, as the library leaves them out of the sort);
  * pooled outputs: sampled bags (and the longest one), each through the oracle on its own;
  * updated rows and Adagrad state: the hottest rows, a random sample of touched rows and a few
    rows no lookup touched, each through the oracle on the lookups that hit it.
"""
from types import SimpleNamespace

import numpy as np
import pytest
import torch

import oracle
from bwd_tbe_fwd_gb300 import TableBatchedEmbedding, TBEOptions
from synth import get_config, make_batch
from synth.gen import grad_out_block, grad_out_tensor, torch_dtype, weight_rows, weights_tensor
from tbe_harness import RTOL, bf16_half_ulp, check_forward, weights_to_oracle

pytestmark = pytest.mark.gpu

N_BAGS = 192    # sampled pooled rows
N_HOT = 8       # hottest rows
N_ROWS = 40     # random touched rows
N_COLD = 4      # rows no lookup touched


def counts_path_tables(cfg):
    """Tables the library runs on the counts x table path with default options (at most 8)."""
    if cfg.wdtype != "f16" or cfg.weighted:
        return []
    return [t for t, spec in enumerate(cfg.tables)
            if spec.histogram and spec.E <= 64 and 64 <= spec.D <= 128][:8]


@pytest.fixture(scope="module", params=["c3", "c5", "c4", "c2"])
def full(request):
    cfg = get_config(request.param)
    batch = make_batch(cfg)
    dev = torch.device("cuda", 0)
    itype = torch.int32 if cfg.itype == "i32" else torch.int64
    opts = TBEOptions(fused_bounds=1)
    tbe = TableBatchedEmbedding(cfg.D, cfg.E, cfg.B, batch.N, torch_dtype(cfg.wdtype), itype,
                                weighted=cfg.weighted, long_bags=[t.histogram for t in cfg.tables],
                                device=dev, options=opts)
    weights = weights_tensor(cfg, device=dev)
    state = (torch.zeros(cfg.total_rows, dtype=torch.float32, device=dev)
             if cfg.optimizer == "adagrad" else None)
    grad = grad_out_tensor(cfg, device=dev)
    idx = torch.from_numpy(batch.indices).to(dev)
    off = torch.from_numpy(batch.offsets).to(dev)
    psw = None if batch.psw is None else torch.from_numpy(batch.psw).to(dev)
    out = torch.empty(cfg.B, cfg.total_D, dtype=torch.float32, device=dev)
    stats = torch.zeros(8, dtype=torch.int64, device=dev)

    # one step, as the benchmark runs it
    tbe.bounds_check(idx, off, stats=stats, offsets_only=True)
    tbe.forward(weights, idx, off, psw=psw, out=out, stats=stats)
    tbe.backward_update(weights, state, idx, off, grad, psw=psw, optimizer=cfg.optimizer, lr=cfg.lr,
                        eps=cfg.eps, stats=stats)
    torch.cuda.synchronize()
    meta = tbe.metadata()

    # the oracle's repair of the host copy, then the host-side linear keys and bag of each lookup
    tables = oracle.Tables(cfg.D, cfg.E)
    idx_h = batch.indices.copy()
    off_h = batch.offsets.copy()
    per_table, n_off = oracle.bounds_repair(tables, cfg.B, idx_h, off_h)
    off64 = off_h.astype(np.int64)
    roff = np.concatenate([[0], np.cumsum(np.asarray(cfg.E, dtype=np.int64))])
    lens = np.diff(off64)
    table_of = np.repeat(np.arange(cfg.T, dtype=np.int64), cfg.B)
    keys = (np.repeat(roff[:-1][table_of], lens) + idx_h.astype(np.int64)).astype(np.int32)
    bag_of = np.repeat(np.arange(cfg.T * cfg.B, dtype=np.int64) % cfg.B, lens)
    # a stable host sort of the keys: every row's lookups (for the updates) and the runs the
    # library must produce (without the counts-path tables' lookups)
    order = np.argsort(keys, kind="stable")
    sk = keys[order]
    head = np.ones(len(sk), dtype=bool)
    head[1:] = sk[1:] != sk[:-1]
    starts = np.flatnonzero(head)
    hist = counts_path_tables(cfg)
    sorted_mask = np.ones(len(keys), dtype=bool)
    for t in hist:
        sorted_mask[off64[t * cfg.B]:off64[(t + 1) * cfg.B]] = False
    ns = SimpleNamespace(cfg=cfg, batch=batch, tbe=tbe, weights=weights, state=state, out=out,
                         stats=stats, meta=meta, idx=idx, off=off, idx_h=idx_h, off_h=off64,
                         per_table=per_table, n_off=n_off, roff=roff, keys=keys, bag_of=bag_of,
                         order=order, sorted_keys=sk, unique=sk[starts],
                         run_off=np.append(starts, len(sk)), sorted_mask=sorted_mask)
    yield ns
    del ns, tbe, weights, state, grad, idx, off, psw, out, stats, meta
    torch.cuda.empty_cache()


def test_full_bounds_repair_is_the_oracles(full):
    assert np.array_equal(full.idx.cpu().numpy(), full.idx_h), "repaired ids differ"
    assert np.array_equal(full.off.cpu().numpy().astype(np.int64), full.off_h), "repaired offsets differ"
    st = full.stats.cpu().numpy()
    assert st[0] == full.per_table.sum() and st[1] == full.n_off


def test_full_run_metadata_bit_exact(full):
    m = full.meta
    keep = full.sorted_mask[full.order]  # the runs of the sort path, in key order
    order = full.order[keep]
    sk = full.sorted_keys[keep]
    N = len(sk)
    assert m["N"] == N
    assert np.array_equal(m["sorted_keys"].cpu().numpy(), sk), "sorted keys differ"
    assert np.array_equal(m["sorted_bags"].cpu().numpy().astype(np.int64), full.bag_of[order]), \
        "sorted bags differ"
    if full.batch.psw is not None and "sorted_psw" in m:
        assert np.array_equal(m["sorted_psw"].cpu().numpy(), full.batch.psw[order]), "sorted psw differ"
    head = np.ones(N, dtype=bool)
    head[1:] = sk[1:] != sk[:-1]
    starts = np.flatnonzero(head)
    run_off = np.append(starts, N)
    assert m["U"] == len(starts)
    assert np.array_equal(m["unique_keys"].cpu().numpy(), sk[starts]), "unique keys differ"
    assert np.array_equal(m["run_offsets"].cpu().numpy().astype(np.int64), run_off), "run offsets differ"
    assert np.array_equal(m["run_lengths"].cpu().numpy().astype(np.int64), np.diff(run_off)), \
        "run lengths differ"


def test_full_forward_sampled_bags(full):
    cfg, B = full.cfg, full.cfg.B
    rng = np.random.default_rng(11)
    lens = np.diff(full.off_h)
    longest = int(np.argmax(lens))
    picks = list(zip(rng.integers(0, cfg.T, N_BAGS).tolist(), rng.integers(0, B, N_BAGS).tolist()))
    picks.append((longest // B, longest % B))
    rows = full.out[torch.tensor([b for _, b in picks], device=full.out.device)].cpu().numpy()
    cols = np.concatenate([[0], np.cumsum(cfg.D)])
    for k, (t, b) in enumerate(picks):
        s, e = int(full.off_h[t * B + b]), int(full.off_h[t * B + b + 1])
        uniq, inv = np.unique(full.idx_h[s:e].astype(np.int64), return_inverse=True)
        if len(uniq) == 0:
            uniq = np.zeros(1, np.int64)
        D = int(cfg.D[t])
        w = weights_to_oracle(weight_rows(cfg, t, uniq).reshape(-1), cfg.wdtype)
        psw = None if full.batch.psw is None else full.batch.psw[s:e]
        _, exact, absterms = oracle.forward(oracle.Tables([D], [len(uniq)]), 1, w, inv.astype(np.int64),
                                            np.array([0, e - s], np.int64), psw=psw, wdtype=cfg.wdtype)
        check_forward(rows[k:k + 1, cols[t]:cols[t] + D], exact, absterms, cfg.wdtype)


def test_full_update_sampled_rows(full):
    cfg = full.cfg
    rtol = RTOL[cfg.wdtype]
    lens = np.diff(full.run_off)
    rng = np.random.default_rng(12)
    runs = np.concatenate([np.argsort(lens)[::-1][:N_HOT], rng.choice(len(lens), N_ROWS, replace=False)])
    eoff = np.asarray(cfg.elem_offsets, dtype=np.int64)
    cols = np.concatenate([[0], np.cumsum(cfg.D)])
    w_gpu = full.weights
    for u in runs.tolist():
        key = int(full.unique[u])
        t = int(np.searchsorted(full.roff, key, side="right") - 1)
        r = key - int(full.roff[t])
        D = int(cfg.D[t])
        pos = full.order[full.run_off[u]:full.run_off[u + 1]]
        bags = full.bag_of[pos]
        n = len(pos)
        # the row's lookups as n one-lookup bags of a one-row table: the same sum of gradients
        g = grad_out_block(cfg, bags, int(cols[t]), D).numpy()
        w = weights_to_oracle(weight_rows(cfg, t, [r]).reshape(-1), cfg.wdtype)
        st = np.zeros(1, np.float32) if cfg.optimizer == "adagrad" else None
        psw = None if full.batch.psw is None else full.batch.psw[pos]
        res = oracle.backward(oracle.Tables([D], [1]), n, w, st, np.zeros(n, np.int64),
                              np.arange(n + 1, dtype=np.int64), g, psw=psw, optimizer=cfg.optimizer,
                              lr=cfg.lr, eps=cfg.eps, wdtype=cfg.wdtype)
        ref = res["w_exact"]
        base = int(eoff[t]) + r * D
        x = w_gpu[base:base + D].to(torch.float64).cpu().numpy()
        bound = rtol * np.maximum(np.abs(ref), np.abs(ref).max() / 64.0)
        if cfg.wdtype == "bf16":
            bound = bound + bf16_half_ulp(ref)
        err = np.abs(x - ref)
        assert (err <= bound).all(), (f"row {r} of table {t} ({n} lookups): element {int(np.argmax(err - bound))} "
                                      f"gpu {x[np.argmax(err - bound)]!r} oracle {ref[np.argmax(err - bound)]!r}")
        if full.state is not None:
            sx = float(full.state[key].item())
            sr = float(res["state_exact"][0])
            assert abs(sx - sr) <= rtol * max(sr, 1e-30), (key, sx, sr)
    # rows no lookup touched: unchanged, bit for bit, and their state still zero
    touched = np.zeros(int(full.roff[-1]), dtype=bool)
    touched[full.unique.astype(np.int64)] = True
    cold = rng.choice(np.flatnonzero(~touched), N_COLD, replace=False)
    for key in cold.tolist():
        t = int(np.searchsorted(full.roff, key, side="right") - 1)
        r = key - int(full.roff[t])
        D = int(cfg.D[t])
        base = int(eoff[t]) + r * D
        x = w_gpu[base:base + D].cpu()
        assert torch.equal(x, weight_rows(cfg, t, [r]).reshape(-1)), f"untouched row {r} of table {t} was written"
        if full.state is not None:
            assert float(full.state[key].item()) == 0.0
