"""Checks that pin the CPU oracle to something other than itself.

Each check takes an ``oracle.Oracle`` (the default build, or a deliberately broken copy in
the mutation tests) and raises AssertionError when the oracle disagrees with:
  * the IEEE-754 definitions of the storage types (numpy's and torch's conversions, and the
    round-to-nearest-even property itself),
  * library routines that compute the same thing by other means: torch's
    ``embedding_bag(mode="sum", per_sample_weights=...)`` for the forward (the reference the
    tutorial chapter checks its kernels against) and torch autograd of it for the SGD backward,
    numpy's stable sort / unique / scatter-add for the run metadata and gradient sums,
  * printed results of the pages' worked examples (tests/golden/, each file cites its source),
  * closed forms and special cases (single-id bags, empty bags, duplicates, routing extremes).
"""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle as oracle_mod
from synth import examples

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ------------------------------------------------------------------------------------------
# helpers (test-side views of the inputs; no oracle arithmetic)
# ------------------------------------------------------------------------------------------
def read_golden(name: str) -> dict:
    rows = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, *vals = line.split()
            rows.setdefault(key, []).append([float(v) for v in vals])
    return rows


def weights_as_f64(w: np.ndarray, wdtype: str) -> np.ndarray:
    if wdtype == "bf16":
        return torch.from_numpy(w.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    return w.astype(np.float64)


def to_storage(w64: np.ndarray, wdtype: str) -> np.ndarray:
    """fp64 -> storage array as the oracle expects it (bf16 as uint16 bits).  The values used
    with this are exactly representable, so the conversion route does not matter."""
    if wdtype == "f32":
        return w64.astype(np.float32)
    if wdtype == "f16":
        return w64.astype(np.float16)
    t = torch.from_numpy(w64.astype(np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def random_problem(rng: np.random.Generator, wdtype: str, T: int = 3, B: int = 7,
                   weighted: bool = False, itype=np.int64, max_len: int = 9, dup_hot: bool = True):
    D = rng.choice([4, 8, 12, 16], size=T).astype(np.int32)
    E = rng.integers(3, 11, size=T).astype(np.int64)
    lengths = rng.integers(0, max_len + 1, size=T * B)
    lengths[rng.random(T * B) < 0.15] = 0                       # some empty bags
    offsets = np.zeros(T * B + 1, dtype=np.int64)
    np.cumsum(lengths, out=offsets[1:])
    N = int(offsets[-1])
    idx = np.empty(N, dtype=np.int64)
    for t in range(T):
        s, e = offsets[t * B], offsets[(t + 1) * B]
        ids = rng.integers(0, E[t], size=e - s)
        if dup_hot:
            ids[rng.random(e - s) < 0.4] = 0                    # a hot row: long runs, duplicates
        idx[s:e] = ids
    elems = int((E * D).sum())
    w64 = np.round(rng.uniform(-1, 1, elems) * 64) / 64         # exactly representable in all dtypes
    w = to_storage(w64, wdtype)
    psw = (np.round(rng.uniform(0, 1, N) * 256) / 256).astype(np.float32) if weighted else None
    grad = rng.standard_normal((B, int(D.sum()))).astype(np.float32)
    return dict(tables=oracle_mod.Tables(D, E), D=D, E=E, B=B, offsets=offsets.astype(itype),
                indices=idx.astype(itype), weights=w, wdtype=wdtype, psw=psw, grad=grad)


def _col_begin(D):
    return np.concatenate([[0], np.cumsum(D)]).astype(np.int64)


def _elem_begin(D, E):
    return np.concatenate([[0], np.cumsum(E * D.astype(np.int64))]).astype(np.int64)


def _table_weight_view(P, t, w64):
    eb = _elem_begin(P["D"], P["E"])
    return w64[eb[t]:eb[t + 1]].reshape(int(P["E"][t]), int(P["D"][t]))


def embedding_bag_reference(P, w64: np.ndarray, mode: str = "sum") -> np.ndarray:
    """Per-table torch embedding_bag (sum, or mean for unweighted problems) in fp64,
    concatenated along columns."""
    B, T = P["B"], P["tables"].T
    offs = P["offsets"].astype(np.int64)
    idx = torch.from_numpy(P["indices"].astype(np.int64))
    outs = []
    for t in range(T):
        o = offs[t * B:(t + 1) * B + 1]
        tab = torch.from_numpy(_table_weight_view(P, t, w64))
        psw = None if P["psw"] is None else torch.from_numpy(P["psw"][o[0]:o[-1]].astype(np.float64))
        outs.append(torch.nn.functional.embedding_bag(
            idx[o[0]:o[-1]], tab, torch.from_numpy(o[:-1] - o[0]), mode=mode, per_sample_weights=psw))
    return torch.cat(outs, dim=1).numpy()


def bag_lengths_per_output(P) -> np.ndarray:
    """[B, sum D]: the length of the bag each output element pools."""
    B, D = P["B"], P["D"]
    L = np.diff(P["offsets"].astype(np.int64)).reshape(len(D), B)
    return np.concatenate([np.repeat(L[t][:, None], D[t], axis=1) for t in range(len(D))], axis=1)


def autograd_psw_grad(P, w64: np.ndarray) -> np.ndarray:
    """d(sum(out * grad_out))/d psw through torch autograd of embedding_bag(mode="sum") in fp64."""
    B, T = P["B"], P["tables"].T
    offs = P["offsets"].astype(np.int64)
    idx = torch.from_numpy(P["indices"].astype(np.int64))
    cb = _col_begin(P["D"])
    out_g = np.full(len(P["indices"]), np.nan)
    for t in range(T):
        o = offs[t * B:(t + 1) * B + 1]
        tab = torch.from_numpy(_table_weight_view(P, t, w64).copy())
        psw = torch.from_numpy(P["psw"][o[0]:o[-1]].astype(np.float64)).requires_grad_(True)
        out = torch.nn.functional.embedding_bag(
            idx[o[0]:o[-1]], tab, torch.from_numpy(o[:-1] - o[0]), mode="sum", per_sample_weights=psw)
        out.backward(torch.from_numpy(P["grad"][:, cb[t]:cb[t + 1]].astype(np.float64)))
        out_g[o[0]:o[-1]] = psw.grad.numpy()
    return out_g


def autograd_weight_grad_mean(P, w64: np.ndarray) -> np.ndarray:
    """As autograd_weight_grad, through embedding_bag(mode="mean") (unweighted)."""
    B, T = P["B"], P["tables"].T
    offs = P["offsets"].astype(np.int64)
    idx = torch.from_numpy(P["indices"].astype(np.int64))
    eb = _elem_begin(P["D"], P["E"])
    grads = np.zeros_like(w64)
    cb = _col_begin(P["D"])
    for t in range(T):
        o = offs[t * B:(t + 1) * B + 1]
        tab = torch.from_numpy(_table_weight_view(P, t, w64).copy()).requires_grad_(True)
        out = torch.nn.functional.embedding_bag(
            idx[o[0]:o[-1]], tab, torch.from_numpy(o[:-1] - o[0]), mode="mean")
        out.backward(torch.from_numpy(P["grad"][:, cb[t]:cb[t + 1]].astype(np.float64)))
        grads[eb[t]:eb[t + 1]] = tab.grad.numpy().reshape(-1)
    return grads


def autograd_weight_grad(P, w64: np.ndarray) -> np.ndarray:
    """d(sum(out * grad_out))/dW through torch autograd of the embedding_bag reference (fp64),
    in the packed layout."""
    B, T = P["B"], P["tables"].T
    offs = P["offsets"].astype(np.int64)
    idx = torch.from_numpy(P["indices"].astype(np.int64))
    eb = _elem_begin(P["D"], P["E"])
    grads = np.zeros_like(w64)
    cb = _col_begin(P["D"])
    for t in range(T):
        o = offs[t * B:(t + 1) * B + 1]
        tab = torch.from_numpy(_table_weight_view(P, t, w64).copy()).requires_grad_(True)
        psw = None if P["psw"] is None else torch.from_numpy(P["psw"][o[0]:o[-1]].astype(np.float64))
        out = torch.nn.functional.embedding_bag(
            idx[o[0]:o[-1]], tab, torch.from_numpy(o[:-1] - o[0]), mode="sum", per_sample_weights=psw)
        g = torch.from_numpy(P["grad"][:, cb[t]:cb[t + 1]].astype(np.float64))
        out.backward(g)
        grads[eb[t]:eb[t + 1]] = tab.grad.numpy().reshape(-1)
    return grads


def lookup_keys_and_bags(P):
    """Linear key and bag of every lookup, in lookup order (table-major offsets)."""
    B, T = P["B"], P["tables"].T
    offs = P["offsets"].astype(np.int64)
    rb = np.concatenate([[0], np.cumsum(P["E"])])
    lengths = np.diff(offs)
    bag_flat = np.repeat(np.arange(T * B), lengths)
    t = bag_flat // B
    b = bag_flat % B
    keys = rb[t] + P["indices"].astype(np.int64)
    return keys, b, t


# ------------------------------------------------------------------------------------------
# checks
# ------------------------------------------------------------------------------------------
def check_half_conversions(orc):
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([orc.half_to_double(int(b)) for b in bits])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    m = ~np.isnan(ref)
    assert np.array_equal(got[m], ref[m]), "fp16 decode"
    # encode: every finite half, every midpoint between neighbours (ties), random magnitudes
    finite = ref[np.isfinite(ref)]
    pos = np.unique(np.abs(finite))
    mids = (pos[:-1] + pos[1:]) / 2
    rng = np.random.default_rng(5)
    rand = rng.standard_normal(4000) * np.exp2(rng.integers(-30, 18, 4000))
    xs = np.concatenate([finite, mids, -mids, rand, [65504.0, 65519.99, 65520.0, 1e6, 2.0 ** -25,
                                                     2.0 ** -25 * 1.0000001, 2.0 ** -26]])
    with np.errstate(over="ignore"):
        want = xs.astype(np.float16).view(np.uint16)
    got = np.array([orc.double_to_half(float(x)) for x in xs], dtype=np.uint16)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, f"fp16 encode of {xs[bad[:5]]}: {got[bad[:5]]} vs {want[bad[:5]]}"


def check_bf16_conversions(orc):
    bits = np.arange(65536, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([orc.bf16_to_double(int(b)) for b in bits])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    m = ~np.isnan(ref)
    assert np.array_equal(got[m], ref[m]), "bf16 decode"
    # encode of float32-representable values: compare with torch's fp32 -> bf16 (RNE)
    rng = np.random.default_rng(6)
    x32 = (rng.standard_normal(6000) * np.exp2(rng.integers(-130, 120, 6000))).astype(np.float32)
    fin = ref[np.isfinite(ref)]
    pos = np.unique(np.abs(fin))
    mids32 = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)     # exact ties are fp32-representable
    x32 = np.concatenate([x32, mids32, -mids32])
    want = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([orc.double_to_bf16(float(x)) for x in x32], dtype=np.uint16)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, f"bf16 encode of {x32[bad[:5]]}"
    # encode of general doubles: the result is a nearest bf16, ties to an even fraction
    xs = rng.standard_normal(3000) * np.exp2(rng.integers(-60, 60, 3000))
    for x in xs:
        r = orc.double_to_bf16(float(x))
        v = orc.bf16_to_double(r)
        up = orc.bf16_to_double((r + 1) & 0xFFFF)
        dn = orc.bf16_to_double((r - 1) & 0xFFFF)
        for nb in (up, dn):
            if np.isfinite(nb) and np.sign(nb) == np.sign(v):
                assert abs(x - v) <= abs(x - nb), f"bf16 not nearest for {x!r}"
                if abs(x - v) == abs(x - nb):
                    assert r % 2 == 0, "bf16 tie not to even"


def check_forward_embedding_bag(orc):
    rng = np.random.default_rng(11)
    for wdtype in ("f32", "f16", "bf16"):
        for weighted in (False, True):
            for itype in (np.int32, np.int64):
                P = random_problem(rng, wdtype, weighted=weighted, itype=itype)
                w64 = weights_as_f64(P["weights"], wdtype)
                out, exact, absterms = orc.forward(P["tables"], P["B"], P["weights"], P["indices"],
                                                   P["offsets"], psw=P["psw"], wdtype=wdtype)
                ref = embedding_bag_reference(P, w64)
                assert np.all(np.abs(exact - ref) <= 1e-12 * np.maximum(absterms, 1e-300)), \
                    f"forward vs embedding_bag ({wdtype}, weighted={weighted})"
                assert np.array_equal(out, exact.astype(np.float32))
                if P["psw"] is None:
                    # absterms of an unweighted bag is the sum of |w|, checked with embedding_bag
                    Q = dict(P)
                    ref_abs = embedding_bag_reference(Q, np.abs(w64))
                    assert np.allclose(absterms, ref_abs, rtol=1e-12, atol=0)


def check_forward_mean(orc):
    """Mean pooling ([TUT], "Try this"): embedding_bag(mode="mean") for unweighted bags (an
    empty bag gives 0 there too); for weighted bags the closed form sum(psw * w) / L, with the
    sum from embedding_bag(mode="sum", per_sample_weights)."""
    rng = np.random.default_rng(21)
    for wdtype in ("f32", "f16", "bf16"):
        for weighted in (False, True):
            P = random_problem(rng, wdtype, weighted=weighted)
            w64 = weights_as_f64(P["weights"], wdtype)
            _, exact, absterms = orc.forward(P["tables"], P["B"], P["weights"], P["indices"], P["offsets"],
                                             psw=P["psw"], wdtype=wdtype, pooling="mean")
            if weighted:
                L = bag_lengths_per_output(P)
                ref = embedding_bag_reference(P, w64) / np.maximum(L, 1)
            else:
                ref = embedding_bag_reference(P, w64, mode="mean")
            assert np.all(np.abs(exact - ref) <= 1e-12 * np.maximum(absterms, 1e-300)), \
                f"mean forward ({wdtype}, weighted={weighted})"


def check_backward_mean_sgd_autograd(orc):
    """SGD with mean pooling equals W - lr * autograd of embedding_bag(mode="mean"); the
    recorded per-lookup factor is 1 / L."""
    rng = np.random.default_rng(22)
    for wdtype in ("f32", "bf16"):
        P = random_problem(rng, wdtype)
        w64 = weights_as_f64(P["weights"], wdtype)
        w = P["weights"].copy()
        lr = 0.125
        res = orc.backward(P["tables"], P["B"], w, None, P["indices"], P["offsets"], P["grad"],
                           optimizer="sgd", lr=lr, wdtype=wdtype, pooling="mean")
        gW = autograd_weight_grad_mean(P, w64)
        expected = w64 - lr * gW
        eb = _elem_begin(P["D"], P["E"])
        rb = np.concatenate([[0], np.cumsum(P["E"])])
        for r, key in enumerate(res["unique_keys"]):
            t = int(np.searchsorted(rb, key, side="right") - 1)
            base = eb[t] + (key - rb[t]) * P["D"][t]
            got = res["w_exact"][res["run_elem_offsets"][r]:res["run_elem_offsets"][r + 1]]
            want = expected[base:base + P["D"][t]]
            assert np.all(np.abs(got - want) <= 1e-12 * (np.abs(want) + lr * np.abs(gW[base:base + P["D"][t]]) + 1e-300)), \
                f"mean SGD vs autograd ({wdtype})"
        # factor of each sorted lookup = 1 / (length of its bag)
        L = np.diff(P["offsets"].astype(np.int64))
        tab_of = np.searchsorted(rb, res["sorted_keys"], side="right") - 1
        want_f = (1.0 / L[tab_of * P["B"] + res["sorted_bags"]]).astype(np.float32)
        assert np.array_equal(res["sorted_psw"], want_f), "mean factor 1/L"


def check_psw_gradient_autograd(orc):
    """Gradient with respect to the per-sample weights: torch autograd of
    embedding_bag(mode="sum", per_sample_weights) in fp64; for mean pooling the same over L."""
    rng = np.random.default_rng(23)
    for wdtype in ("f32", "f16", "bf16"):
        P = random_problem(rng, wdtype, weighted=True)
        w64 = weights_as_f64(P["weights"], wdtype)
        g = orc.psw_gradient(P["tables"], P["B"], P["weights"], P["indices"], P["offsets"], P["grad"],
                             wdtype=wdtype)
        ref = autograd_psw_grad(P, w64)
        assert np.all(np.abs(g - ref) <= 1e-12 * (np.abs(ref) + 1e-9)), f"psw gradient ({wdtype})"
        gm = orc.psw_gradient(P["tables"], P["B"], P["weights"], P["indices"], P["offsets"], P["grad"],
                              wdtype=wdtype, pooling="mean")
        Ls = np.concatenate([np.full(int(n), float(n)) for n in np.diff(P["offsets"].astype(np.int64))])
        assert np.all(np.abs(gm - ref / Ls) <= 1e-12 * (np.abs(ref) + 1e-9)), f"mean psw gradient ({wdtype})"


def check_forward_special_cases(orc):
    # T=2 tables: D=(4, 8), E=(5, 3); bags chosen by hand
    D = np.array([4, 8], np.int32)
    E = np.array([5, 3], np.int64)
    tables = oracle_mod.Tables(D, E)
    B = 3
    w64 = np.arange(int((E * D).sum()), dtype=np.float64) / 8.0 - 3.0
    w = w64.astype(np.float32)
    # table 0: bag0=[2], bag1=[], bag2=[4,4,4]; table 1: bag0=[], bag1=[1,0], bag2=[2]
    bags = [[2], [], [4, 4, 4], [], [1, 0], [2]]
    offsets = np.concatenate([[0], np.cumsum([len(b) for b in bags])]).astype(np.int64)
    idx = np.array([i for b in bags for i in b], dtype=np.int64)
    out, exact, _ = orc.forward(tables, B, w, idx, offsets)
    row = lambda t, i: w64[[0, 20][t] + i * D[t]:[0, 20][t] + (i + 1) * D[t]]  # noqa: E731
    want = np.zeros((B, 12))
    want[0, :4] = row(0, 2)
    want[2, :4] = 3 * row(0, 4)
    want[1, 4:] = row(1, 1) + row(1, 0)
    want[2, 4:] = row(1, 2)
    assert np.array_equal(exact, want), "single / empty / duplicate bags"
    # weights scale each lookup: doubling psw doubles the output
    psw = np.full(idx.shape, 0.5, np.float32)
    _, e1, _ = orc.forward(tables, B, w, idx, offsets, psw=psw)
    _, e2, _ = orc.forward(tables, B, w, idx, offsets, psw=2 * psw)
    assert np.array_equal(e1 * 2, e2) and np.array_equal(e1, 0.5 * want)


def check_backward_sgd_autograd(orc):
    rng = np.random.default_rng(12)
    for wdtype in ("f32", "f16", "bf16"):
        for weighted in (False, True):
            P = random_problem(rng, wdtype, weighted=weighted)
            w64 = weights_as_f64(P["weights"], wdtype)
            w = P["weights"].copy()
            lr = 0.125
            res = orc.backward(P["tables"], P["B"], w, None, P["indices"], P["offsets"], P["grad"],
                               psw=P["psw"], optimizer="sgd", lr=lr, wdtype=wdtype)
            gW = autograd_weight_grad(P, w64)
            expected = w64 - lr * gW
            # touched elements: the run of each unique key
            eb = _elem_begin(P["D"], P["E"])
            rb = np.concatenate([[0], np.cumsum(P["E"])])
            touched = np.zeros(w64.shape, bool)
            got_exact = np.empty(w64.shape)
            for r, key in enumerate(res["unique_keys"]):
                t = int(np.searchsorted(rb, key, side="right") - 1)
                base = eb[t] + (key - rb[t]) * P["D"][t]
                sl = slice(base, base + P["D"][t])
                touched[sl] = True
                got_exact[sl] = res["w_exact"][res["run_elem_offsets"][r]:res["run_elem_offsets"][r + 1]]
            scale = np.abs(w64) + lr * np.abs(gW) + 1e-300
            assert np.all(np.abs(got_exact[touched] - expected[touched]) <= 1e-12 * scale[touched]), \
                f"SGD update vs autograd ({wdtype}, weighted={weighted})"
            # every row with a gradient through autograd is a run of the oracle, and the others
            # are left bit-identical
            assert np.all(gW[~touched] == 0), "a row with a gradient has no run"
            assert np.array_equal(weights_as_f64(w, wdtype)[~touched], w64[~touched]), "untouched rows changed"
            assert np.array_equal(weights_as_f64(w, wdtype)[touched],
                                  weights_as_f64(to_storage_rne(expected[touched], wdtype), wdtype))


def to_storage_rne(x64: np.ndarray, wdtype: str) -> np.ndarray:
    """Round-to-nearest-even of fp64 values into the storage type by library conversions
    (numpy for fp32/fp16; fp64 -> bf16 through an exact fp32 split when needed)."""
    if wdtype == "f32":
        return x64.astype(np.float32)
    if wdtype == "f16":
        return x64.astype(np.float16)
    # round to bf16 = round to 8 significant bits, ties to even: use np.float32 arithmetic on
    # values rescaled so that the rounding point is at an integer
    m, e = np.frexp(x64)                      # x = m * 2^e, |m| in [0.5, 1)
    q = np.rint(np.ldexp(m, 8))               # 8 significant bits, ties to even
    v = np.ldexp(q, e - 8)
    return to_storage(v, "bf16")


def check_backward_metadata_library(orc):
    rng = np.random.default_rng(13)
    for itype in (np.int32, np.int64):
        P = random_problem(rng, "f32", weighted=True, itype=itype, T=4, B=9)
        w = P["weights"].copy()
        res = orc.backward(P["tables"], P["B"], w, None, P["indices"], P["offsets"], P["grad"],
                           psw=P["psw"], optimizer="sgd", lr=0.5)
        keys, bags, _ = lookup_keys_and_bags(P)
        order = np.argsort(keys, kind="stable")
        assert np.array_equal(res["sorted_keys"], keys[order]), "sorted keys"
        assert np.array_equal(res["sorted_bags"], bags[order]), "sorted payload order"
        assert np.array_equal(res["sorted_psw"], P["psw"][order]), "sorted psw"
        uk, cnt = np.unique(keys, return_counts=True)
        assert np.array_equal(res["unique_keys"], uk) and np.array_equal(res["run_lengths"], cnt)
        assert np.array_equal(res["run_offsets"], np.concatenate([[0], np.cumsum(cnt)]))
        assert res["num_lookups"] == len(keys) and int(res["run_lengths"].sum()) == len(keys)


def check_grad_sum_scatter(orc):
    rng = np.random.default_rng(14)
    P = random_problem(rng, "f16", weighted=True, T=3, B=11)
    w = P["weights"].copy()
    res = orc.backward(P["tables"], P["B"], w, None, P["indices"], P["offsets"], P["grad"],
                       psw=P["psw"], optimizer="sgd", lr=0.0, wdtype="f16")
    keys, bags, tabs = lookup_keys_and_bags(P)
    cb = _col_begin(P["D"])
    uk = np.unique(keys)
    for r, key in enumerate(uk):
        sel = np.nonzero(keys == key)[0]
        t = tabs[sel[0]]
        rows = P["grad"][bags[sel], cb[t]:cb[t + 1]].astype(np.float64) * P["psw"][sel, None]
        want = np.zeros(P["D"][t])
        np.add.at(want, np.arange(P["D"][t])[None, :].repeat(len(sel), 0), rows)
        got = res["grad_sum"][res["run_elem_offsets"][r]:res["run_elem_offsets"][r + 1]]
        assert np.allclose(got, want, rtol=1e-13, atol=1e-13), "per-row gradient sum"
    # with lr = 0 nothing changes
    assert np.array_equal(w.view(np.uint16), P["weights"].view(np.uint16))


def _adagrad_row_runs(orc, w0, grads, lr, eps, per_lookup: bool):
    D = w0.shape[0]
    tables = oracle_mod.Tables([D], [1])
    w = w0.astype(np.float32).copy()
    state = np.zeros(1, np.float32)
    batches = [[g] for g in grads] if per_lookup else [list(grads)]
    for batch in batches:
        B = len(batch)
        offsets = np.arange(B + 1, dtype=np.int64)
        idx = np.zeros(B, dtype=np.int64)
        orc.backward(tables, B, w, state, idx, offsets, np.stack(batch), optimizer="adagrad",
                     lr=lr, eps=eps)
    return w


def check_adagrad_golden(orc):
    gold = read_golden("adagrad_trap.txt")
    w0, grads, lr, eps = examples.adagrad_trap_inputs()
    one = _adagrad_row_runs(orc, w0, grads, lr, eps, per_lookup=False)
    five = _adagrad_row_runs(orc, w0, grads, lr, eps, per_lookup=True)
    assert np.all(np.abs(one - np.array(gold["one_step_summed"][0])) <= 5e-5), f"one step: {one}"
    assert np.all(np.abs(five - np.array(gold["five_per_lookup"][0])) <= 5e-5), f"five steps: {five}"
    assert abs(float(np.abs(one - five).max()) - gold["max_abs_difference"][0][0]) <= 5e-4


def check_skewed_batch_golden(orc):
    gold = read_golden("skewed_batch_runs.txt")
    ex = examples.skewed_batch(seed=1)
    T, E, B, D = ex["T"], ex["E"], ex["B"], ex["D"]
    tables = oracle_mod.Tables([D] * T, [E] * T)
    grad = examples.skewed_batch_grad(B, T * D)
    w = ex["W"].reshape(-1).copy()
    res = orc.backward(tables, B, w, None, ex["indices"], ex["offsets"], grad, optimizer="sgd", lr=0.05)
    assert res["num_lookups"] == gold["lookups"][0][0]
    assert res["num_runs"] == gold["unique_rows"][0][0]
    assert int(res["run_lengths"].max()) == gold["max_run"][0][0]
    for thr, chunk, n_short, n_long, n_chunks in gold["sweep"]:
        c = orc.classify(tables, res["unique_keys"], res["run_lengths"], int(thr), int(chunk))
        assert (c["num_short"], c["num_long"], c["num_chunks"]) == (n_short, n_long, n_chunks), \
            f"sweep {thr},{chunk}: {c['num_short']},{c['num_long']},{c['num_chunks']}"
    # and the update itself is W - lr * autograd gradient of the embedding_bag reference
    P = dict(tables=tables, D=np.array([D] * T, np.int32), E=np.array([E] * T, np.int64), B=B,
             offsets=ex["offsets"], indices=ex["indices"], psw=None, grad=grad)
    gW = autograd_weight_grad(P, ex["W"].reshape(-1).astype(np.float64))
    want = ex["W"].reshape(-1).astype(np.float64) - 0.05 * gW
    assert np.allclose(w.astype(np.float64), want, rtol=0, atol=1e-7)


def check_bounds_repair(orc):
    D = np.array([4, 4], np.int32)
    E = np.array([5, 3], np.int64)
    tables = oracle_mod.Tables(D, E)
    B = 3
    # valid input: nothing changes
    offsets = np.array([0, 2, 2, 5, 6, 6, 8], np.int64)
    idx = np.array([0, 4, 1, 2, 3, 0, 1, 2], np.int64)
    o2, i2 = offsets.copy(), idx.copy()
    per, noff = orc.bounds_repair(tables, B, i2, o2)
    assert noff == 0 and per.tolist() == [0, 0] and np.array_equal(o2, offsets) and np.array_equal(i2, idx)
    # bad ids: negative, == E, > E; each becomes 0 and is counted in its own table
    idx_bad = np.array([-1, 5, 1, 7, 3, 0, 3, -9], np.int64)
    per, noff = orc.bounds_repair(tables, B, idx_bad, offsets.copy())
    assert per.tolist() == [3, 2] and noff == 0
    assert idx_bad.tolist() == [0, 0, 1, 0, 3, 0, 0, 0]
    # offsets: first not 0, a decrease, one above the last, last above num_indices
    off_bad = np.array([1, 5, 3, 9, 6, 6, 12], np.int64)
    i3 = idx.copy()
    per, noff = orc.bounds_repair(tables, B, i3, off_bad, num_indices=8)
    assert off_bad.tolist() == [0, 5, 5, 8, 8, 8, 8], off_bad.tolist()
    assert noff == 6  # last, first, and offsets 2, 3, 4, 5
    for itype in (np.int32,):
        o4 = offsets.astype(itype)
        i4 = idx_bad.astype(itype)
        orc.bounds_repair(tables, B, i4, o4)
        assert i4.tolist() == [0, 0, 1, 0, 3, 0, 0, 0]


def check_classify(orc):
    rng = np.random.default_rng(15)
    D = np.array([3, 32, 33, 64, 100, 128, 256, 1024], np.int32)
    E = np.array([50, 40, 30, 20, 60, 70, 10, 5], np.int64)
    tables = oracle_mod.Tables(D, E)
    rb = np.concatenate([[0], np.cumsum(E)])
    keys = np.sort(rng.choice(int(rb[-1]), size=200, replace=False)).astype(np.int64)
    lens = rng.integers(1, 700, size=200).astype(np.int64)
    tab = np.searchsorted(rb, keys, side="right") - 1
    bucket = np.ceil(np.log2(D[tab])).astype(int)
    for thr, chunk in [(256, 256), (1, 1), (10 ** 9, 7), (100, 33)]:
        c = orc.classify(tables, keys, lens, thr, chunk)
        is_long = lens >= thr
        assert c["num_long"] == int(is_long.sum())
        assert c["num_chunks"] == int(np.sum(-(-lens[is_long] // chunk)))
        want = np.bincount(bucket[~is_long], minlength=oracle_mod.NUM_BUCKETS)
        assert np.array_equal(c["short_per_bucket"], want)
        assert np.array_equal(c["route"], np.where(is_long, -1, bucket))




def check_adagrad_closed_form(orc):
    """A row touched by one lookup whose gradient row is the constant c has mean(g^2) = c^2,
    so row-wise Adagrad moves every element by lr * c / (|c| + eps) from state 0, and by
    lr * c / (sqrt(2) |c| + eps) on a second identical step (the state accumulates)."""
    D = 8
    tables = oracle_mod.Tables([D], [1])
    lr, eps = 0.5, 1e-8
    for c in (0.75, -3.0, 1e-6, -2e-7):
        w = np.full(D, 0.25, np.float64)
        state = np.zeros(1, np.float32)
        grad = np.full((1, D), c, np.float32)
        c32 = float(np.float32(c))
        for step in (1, 2):
            wf = w.astype(np.float32)
            res = orc.backward(tables, 1, wf, state, np.zeros(1, np.int64), np.array([0, 1], np.int64),
                               grad, optimizer="adagrad", lr=lr, eps=eps)
            want = w - lr * c32 / (np.sqrt(step) * abs(c32) + float(np.float32(eps)))
            assert np.allclose(res["w_exact"], want, rtol=1e-6, atol=0), (c, step, res["w_exact"][0], want[0])
            w = wf.astype(np.float64)


ALL_CHECKS = [
    check_half_conversions,
    check_bf16_conversions,
    check_forward_embedding_bag,
    check_forward_special_cases,
    check_forward_mean,
    check_backward_mean_sgd_autograd,
    check_psw_gradient_autograd,
    check_backward_sgd_autograd,
    check_backward_metadata_library,
    check_grad_sum_scatter,
    check_adagrad_golden,
    check_adagrad_closed_form,
    check_skewed_batch_golden,
    check_bounds_repair,
    check_classify,
]
