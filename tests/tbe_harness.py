"""Shared GPU-test machinery: draw one workload, run the CUDA library through its C-ABI
binding and the CPU oracle on the same bytes, and compare.

Tolerances (stated per element, derived from the arithmetic; the stated maxima are a
relative error of 1e-5 for fp32 tables and 2e-3 for fp16/bf16 tables):
  * pooled output x vs the oracle's unrounded fp64 value r with condition scale S (the sum of
    |psw * w| over the bag):  |x - r| <= rtol * max(|r|, S / 256).  The floor S/256 admits the
    fp32 accumulation error of any summation order on cancelling sums and nothing larger.
  * updated weight x vs the fp64 update r (row of the oracle):  |x - r| <= rtol * max(|r|,
    max_row|r| / 64)  [+ half an ulp of bf16 at r for bf16 tables: bf16 keeps 8 significant
    bits, so its own rounding (up to 2^-8 relative) exceeds 2e-3 by construction].
  * Adagrad state x vs r:  |x - r| <= rtol * r  (all terms are non-negative).
  * rows no lookup touched, and everything integer (repaired ids/offsets, sorted keys, sorted
    bags, unique keys, run offsets/lengths, route counts): bit-exact.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from bwd_tbe_fwd_gb300 import TableBatchedEmbedding, TBEOptions
from synth import make_batch
from synth.gen import grad_out_tensor, weights_tensor

RTOL = {"f32": 1e-5, "f16": 2e-3, "bf16": 2e-3}
TORCH_W = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


def weights_to_oracle(w: torch.Tensor, wdtype: str) -> np.ndarray:
    w = w.detach().cpu().contiguous()
    if wdtype == "bf16":
        return w.view(torch.int16).numpy().view(np.uint16).copy()
    return w.numpy().copy()


def weights_f64(w: torch.Tensor) -> np.ndarray:
    return w.detach().cpu().to(torch.float64).numpy()


def bf16_half_ulp(r: np.ndarray) -> np.ndarray:
    """Half the spacing of bf16 numbers at |r| (normal range; subnormal spacing below it)."""
    a = np.abs(r)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.ldexp(1.0, (e - 8).astype(np.int64))


def check_forward(x: np.ndarray, exact: np.ndarray, absterms: np.ndarray, wdtype: str):
    rtol = RTOL[wdtype]
    err = np.abs(x.astype(np.float64) - exact)
    bound = rtol * np.maximum(np.abs(exact), absterms / 256.0)
    bad = err > bound
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"forward mismatch at {tuple(i)}: gpu {x[tuple(i)]!r} oracle {exact[tuple(i)]!r} "
                             f"({int(bad.sum())} elements out of tolerance)")


def check_update(cfg_tables: oracle.Tables, w_gpu: np.ndarray, w_init: np.ndarray, res: dict, wdtype: str,
                 state_gpu: np.ndarray | None = None, state_init: np.ndarray | None = None):
    """w_gpu / w_init: fp64 views of the whole packed weights after / before."""
    rtol = RTOL[wdtype]
    D, E = cfg_tables.D, cfg_tables.E
    eb = np.concatenate([[0], np.cumsum(E * D.astype(np.int64))])
    rb = np.concatenate([[0], np.cumsum(E)])
    keys = res["unique_keys"]
    t = np.searchsorted(rb, keys, side="right") - 1
    touched = np.zeros(w_gpu.shape, dtype=bool)
    reo = res["run_elem_offsets"]
    for r in range(len(keys)):
        base = eb[t[r]] + (keys[r] - rb[t[r]]) * D[t[r]]
        sl = slice(int(base), int(base + D[t[r]]))
        touched[sl] = True
        ref = res["w_exact"][reo[r]:reo[r + 1]]
        x = w_gpu[sl]
        floor = np.abs(ref).max() / 64.0
        bound = rtol * np.maximum(np.abs(ref), floor)
        if wdtype == "bf16":
            bound = bound + bf16_half_ulp(ref)
        err = np.abs(x - ref)
        if (err > bound).any():
            j = int(np.argmax(err - bound))
            raise AssertionError(f"update mismatch in run {r} (key {keys[r]}, len {res['run_lengths'][r]}), "
                                 f"element {j}: gpu {x[j]!r} oracle {ref[j]!r} bound {bound[j]:.3g}")
    untouched = ~touched
    if not np.array_equal(w_gpu[untouched], w_init[untouched]):
        raise AssertionError("a row no lookup touched was written")
    if state_gpu is not None:
        ref = res["state_exact"]
        x = state_gpu[keys].astype(np.float64)
        bad = np.abs(x - ref) > rtol * np.maximum(ref, 1e-30)
        if bad.any():
            j = int(np.argmax(bad))
            raise AssertionError(f"state mismatch at key {keys[j]}: gpu {x[j]!r} oracle {ref[j]!r}")
        mask = np.ones(state_gpu.shape, dtype=bool)
        mask[keys] = False
        if not np.array_equal(state_gpu[mask], state_init[mask]):
            raise AssertionError("state of an untouched row was written")


class Case:
    """One workload instance on both sides."""

    def __init__(self, cfg, device="cuda", options: TBEOptions | None = None, threshold=None, chunk=None,
                 bounds_check=True, pooling="sum"):
        self.cfg = cfg
        self.pooling = pooling
        self.batch = make_batch(cfg)
        self.tables = oracle.Tables(cfg.D, cfg.E)
        opts = options or TBEOptions()
        if threshold is not None:
            opts.c.long_threshold = threshold
        if chunk is not None:
            opts.c.chunk = chunk
        self.options = opts
        itype = torch.int32 if cfg.itype == "i32" else torch.int64
        self.tbe = TableBatchedEmbedding(
            cfg.D, cfg.E, cfg.B, self.batch.N, TORCH_W[cfg.wdtype], itype, weighted=cfg.weighted,
            long_bags=[t.histogram for t in cfg.tables], device=device, options=opts, pooling=pooling)
        self.device = device
        self.w0 = weights_tensor(cfg)                     # CPU, exact generator values
        self.grad = grad_out_tensor(cfg)                  # CPU [B, sum D]
        # host (oracle) copies
        self.idx_h = self.batch.indices.copy()
        self.off_h = self.batch.offsets.copy()
        # device copies
        self.idx_d = torch.from_numpy(self.batch.indices.copy()).to(device)
        self.off_d = torch.from_numpy(self.batch.offsets.copy()).to(device)
        self.psw_h = self.batch.psw
        self.psw_d = None if self.batch.psw is None else torch.from_numpy(self.batch.psw).to(device)
        self.stats = torch.zeros(8, dtype=torch.int64, device=device)
        self.bounds_checked = False
        if bounds_check:
            self.run_bounds()

    def run_bounds(self):
        per_table, n_off = oracle.bounds_repair(self.tables, self.cfg.B, self.idx_h, self.off_h)
        self.tbe.bounds_check(self.idx_d, self.off_d, stats=self.stats)
        torch.cuda.synchronize()
        assert np.array_equal(self.idx_d.cpu().numpy(), self.idx_h), "repaired ids differ"
        assert np.array_equal(self.off_d.cpu().numpy(), self.off_h), "repaired offsets differ"
        st = self.stats.cpu().numpy()
        assert st[0] == per_table.sum() and st[1] == n_off, (st, per_table.sum(), n_off)
        self.bounds_checked = True
        return per_table, n_off

    def forward(self, options=None):
        w_d = self.w0.to(self.device)
        out = self.tbe.forward(w_d, self.idx_d, self.off_d, psw=self.psw_d, stats=self.stats, options=options)
        torch.cuda.synchronize()
        o_out, exact, absterms = oracle.forward(self.tables, self.cfg.B, weights_to_oracle(self.w0, self.cfg.wdtype),
                                                self.idx_h, self.off_h, psw=self.psw_h, wdtype=self.cfg.wdtype,
                                                pooling=self.pooling)
        check_forward(out.cpu().numpy(), exact, absterms, self.cfg.wdtype)
        return out

    def psw_gradient(self):
        """The library's gradient with respect to the per-sample weights against the oracle's,
        per lookup, within rtol of the sum of |grad * w| over the row (its condition scale)."""
        cfg = self.cfg
        w_d = self.w0.to(self.device)
        g = self.tbe.psw_gradient(w_d, self.idx_d, self.off_d, self.grad.to(self.device))
        torch.cuda.synchronize()
        w_h = weights_to_oracle(self.w0, cfg.wdtype)
        ref = oracle.psw_gradient(self.tables, cfg.B, w_h, self.idx_h, self.off_h, self.grad.numpy(),
                                  wdtype=cfg.wdtype, pooling=self.pooling)
        # condition scale: sum_d |grad * w| of each lookup (over L for mean pooling)
        w64 = weights_f64(self.w0)
        D = np.asarray(cfg.D, dtype=np.int64)
        E = np.asarray(cfg.E, dtype=np.int64)
        eb = np.concatenate([[0], np.cumsum(E * D)])
        cb = np.concatenate([[0], np.cumsum(D)])
        off = self.off_h.astype(np.int64)
        scale = np.zeros(len(ref))
        for t in range(cfg.T):
            for_b = np.repeat(np.arange(cfg.B), np.diff(off[t * cfg.B:(t + 1) * cfg.B + 1]))
            s, e = off[t * cfg.B], off[(t + 1) * cfg.B]
            rows = w64[eb[t]:eb[t + 1]].reshape(E[t], D[t])[self.idx_h[s:e].astype(np.int64)]
            gr = self.grad.numpy()[for_b, cb[t]:cb[t + 1]].astype(np.float64)
            sc = np.abs(rows * gr).sum(axis=1)
            if self.pooling == "mean":
                sc /= np.diff(off[t * cfg.B:(t + 1) * cfg.B + 1])[for_b]
            scale[s:e] = sc
        n = int(off[-1])
        x = g.cpu().numpy()[:n].astype(np.float64)
        err = np.abs(x - ref[:n])
        bad = err > RTOL[cfg.wdtype] * np.maximum(np.abs(ref[:n]), scale[:n]) + 1e-30
        if bad.any():
            i = int(np.argwhere(bad)[0][0])
            raise AssertionError(f"psw gradient mismatch at {i}: gpu {x[i]!r} oracle {ref[i]!r} "
                                 f"({int(bad.sum())} of {n} out of tolerance)")
        return g

    def backward(self, optimizer=None, steps=1, options=None, check_meta=True, prepared=False,
                 reuse_forward=False):
        cfg = self.cfg
        assert steps == 1 or cfg.wdtype == "f32", "multi-step parity needs fp32 tables"
        opt = optimizer or cfg.optimizer
        w_d = self.w0.to(self.device)
        state_d = torch.zeros(cfg.total_rows, dtype=torch.float32, device=self.device) if opt == "adagrad" else None
        w_h = weights_to_oracle(self.w0, cfg.wdtype)
        state_h = np.zeros(cfg.total_rows, dtype=np.float32) if opt == "adagrad" else None
        grad_d = self.grad.to(self.device)
        grad_h = self.grad.numpy()
        res = None
        for step in range(steps):
            w_before = weights_f64(w_d)
            s_before = None if state_d is None else state_d.cpu().numpy().copy()
            if prepared:
                # the transpose on a second stream while the forward gather runs on this one
                main = torch.cuda.current_stream(self.device)
                side = torch.cuda.Stream(device=self.device)
                side.wait_stream(main)
                self.tbe.backward_prepare(self.idx_d, self.off_d, psw=self.psw_d, stats=self.stats, stream=side,
                                          options=options)
                self.tbe.forward(w_d, self.idx_d, self.off_d, psw=self.psw_d)
                main.wait_stream(side)
            self.tbe.backward_update(w_d, state_d, self.idx_d, self.off_d, grad_d, psw=self.psw_d, optimizer=opt,
                                     lr=cfg.lr, eps=cfg.eps, stats=self.stats, options=options, prepared=prepared,
                                     reuse_forward=reuse_forward)
            torch.cuda.synchronize()
            res = oracle.backward(self.tables, cfg.B, w_h, state_h, self.idx_h, self.off_h, grad_h, psw=self.psw_h,
                                  optimizer=opt, lr=cfg.lr, eps=cfg.eps, wdtype=cfg.wdtype, pooling=self.pooling)
            if check_meta:
                self.check_metadata(res, options)
            # each side continues from its own results (the oracle never takes GPU values);
            # over several steps the two trajectories may drift apart by the storage rounding,
            # so multi-step checks use fp32 tables, whose rounding is far below 1e-5
            check_update(self.tables, weights_f64(w_d), w_before, res, cfg.wdtype,
                         None if state_d is None else state_d.cpu().numpy(), s_before)
        return res

    def counts_path_tables(self, options=None):
        """Tables whose backward the library runs as counts^T x grad_out (their lookups are not in
        the sorted metadata): the forward's counts x table tables, at most 8."""
        cfg = self.cfg
        if (not (options or self.options).c.histogram or cfg.wdtype != "f16" or cfg.weighted
                or self.pooling != "sum"):
            return []
        hist = [t for t, spec in enumerate(cfg.tables)
                if spec.E <= 64 and 64 <= spec.D <= 128 and spec.histogram]
        return hist[:8]

    def check_metadata(self, res, options=None):
        m = self.tbe.metadata()
        hist = self.counts_path_tables(options)
        if hist:
            # the oracle's runs without the counts-path tables' rows (keys keep their order)
            roff = np.concatenate([[0], np.cumsum([t.E for t in self.cfg.tables])])
            def keep(keys):
                k = np.ones(len(keys), dtype=bool)
                for t in hist:
                    k &= ~((keys >= roff[t]) & (keys < roff[t + 1]))
                return k
            ks = keep(res["sorted_keys"])
            ku = keep(res["unique_keys"])
            res = dict(res)
            res["sorted_keys"] = res["sorted_keys"][ks]
            res["sorted_bags"] = res["sorted_bags"][ks]
            if "sorted_psw" in res:
                res["sorted_psw"] = res["sorted_psw"][ks]
            res["unique_keys"] = res["unique_keys"][ku]
            res["run_lengths"] = res["run_lengths"][ku]
            res["run_offsets"] = np.concatenate([[0], np.cumsum(res["run_lengths"])]).astype(np.int64)
            res["num_lookups"] = int(ks.sum())
            res["num_runs"] = int(ku.sum())
        N, U = res["num_lookups"], res["num_runs"]
        assert m["N"] == N, (m["N"], N)
        assert m["U"] == U, (m["U"], U)
        assert np.array_equal(m["sorted_keys"].cpu().numpy().astype(np.int64), res["sorted_keys"]), "sorted keys"
        assert np.array_equal(m["sorted_bags"].cpu().numpy().astype(np.int64), res["sorted_bags"]), "sorted bags"
        if "sorted_psw" in m:
            assert np.array_equal(m["sorted_psw"].cpu().numpy(), res["sorted_psw"]), "sorted psw"
        assert np.array_equal(m["unique_keys"].cpu().numpy().astype(np.int64), res["unique_keys"]), "unique keys"
        assert np.array_equal(m["run_offsets"].cpu().numpy().astype(np.int64), res["run_offsets"]), "run offsets"
        assert np.array_equal(m["run_lengths"].cpu().numpy().astype(np.int64), res["run_lengths"]), "run lengths"
        c = oracle.classify(self.tables, res["unique_keys"], res["run_lengths"], self.options.c.long_threshold,
                            self.options.c.chunk)
        assert m["num_long"] == c["num_long"] and m["num_chunks"] == c["num_chunks"], \
            (m["num_long"], c["num_long"], m["num_chunks"], c["num_chunks"])
        assert np.array_equal(m["short_per_bucket"].astype(np.int64), c["short_per_bucket"]), \
            (m["short_per_bucket"], c["short_per_bucket"])
        return m, c
