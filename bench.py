#!/usr/bin/env python
"""Benchmark of one table-batched-embedding training step on GB300.

A step is the whole hot path over one batch: bounds check + pooled forward + backward with
one row-wise Adagrad update per touched row (tbe_bounds_check, tbe_forward,
tbe_backward_update through the C-ABI).  The default workload is the large skew stress batch
(T=32 tables of 4M fp16 rows x 128, B=131072, ~83.9M lookups, ~3M distinct rows, hottest
row ~125K hits), drawn by `synth` on the host; weights and upstream gradients are generated
on the device by the same counter-based generator the checks use.

Prints ONE JSON line (rank 0).  `--impl reference` times the CPU oracle instead (bounded
samples of the same workload, single-threaded), as the reference arm.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "TBE fwd+bwd lookups/s and achieved HBM GB/s (% of roofline) on 1 GB300"
FALLBACK_HBM_GBS = 6800.0
BOUNDS_LAUNCHES = {"separate": 3, "fused": 2}  # offsets max, offsets fix (+ ids check)


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=60)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="c3", help="workload: c1..c5 (default c3, the large skew batch)")
    ap.add_argument("--long-mode", choices=["auto", "two_kernel", "fused"], default="auto")
    ap.add_argument("--scheduler", choices=["grid", "persistent", "clc"], default="persistent")
    ap.add_argument("--merge", choices=["atomic", "bulk"], default="atomic")
    ap.add_argument("--gather", choices=["register", "tma"], default="register",
                    help="forward row gather: tma = tile::gather4 copies (equal-width 16-bit tables)")
    ap.add_argument("--pooling", choices=["sum", "mean"], default="sum")
    ap.add_argument("--bounds", choices=["fused", "separate"], default="fused",
                    help="fused: the offsets kernel, then the forward repairs ids as it reads them; "
                         "separate: tbe_bounds_check repairs offsets and ids before the forward")
    ap.add_argument("--psw-grad", action="store_true",
                    help="weighted workloads: also compute the gradient with respect to the per-sample "
                         "weights (tbe_psw_gradient) in each step, before the update")
    ap.add_argument("--classify", choices=["atomic", "ordered"], default="ordered")
    ap.add_argument("--hoist", choices=["on", "off"], default="off",
                    help="run the backward's transpose (tbe_backward_prepare) on a second stream beside "
                         "the forward gather")
    ap.add_argument("--reuse-counts", choices=["on", "off"], default="on",
                    help="the backward of the counts x table tables takes the per-bag counts the forward "
                         "of the same step saved (tbe_options.forward_ws) instead of reading the ids again")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-side", action="store_true",
                    help="skip the side measurement of the other run classifier (a few steps of the "
                         "headline workload with --classify flipped)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--tables", type=int, default=0,
                    help="keep only the first T tables of the workload (small cases for profiling)")
    ap.add_argument("--bags", type=int, default=0,
                    help="bags per table (B) of the workload (small cases for profiling)")
    ap.add_argument("--per-config", default="c1,c2,c4,c5",
                    help="comma-separated other workloads timed after the headline one (empty: none)")
    ap.add_argument("--cpu-sample-bags", type=int, default=0,
                    help="bags per table in the CPU oracle sample (0: sized for ~15 s)")
    return ap.parse_args()


# ------------------------------------------------------------------------------------------
# distributed helpers (replicas only: no data-path collective)
# ------------------------------------------------------------------------------------------
def dist_setup(backend):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    if backend == "nccl":
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def all_max(world, x: float, device) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def all_sum(world, x: float, device) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------------------------------------
# workload statistics and algorithmic bytes
# ------------------------------------------------------------------------------------------
def batch_stats(cfg, batch):
    """Per-lookup keys -> runs on the host (numpy), for the byte model and the JSON line."""
    T, B = cfg.T, cfg.B
    off = batch.offsets.astype(np.int64)
    per_table = np.array([off[(t + 1) * B] - off[t * B] for t in range(T)], dtype=np.int64)
    rb = np.concatenate([[0], np.cumsum(cfg.E)])
    tab = np.repeat(np.arange(T), per_table)
    idx = batch.indices.astype(np.int64)
    valid = (idx >= 0) & (idx < cfg.E[tab])
    keys = rb[tab] + np.where(valid, idx, 0)
    uk, cnt = np.unique(keys, return_counts=True)
    utab = np.searchsorted(rb, uk, side="right") - 1
    return dict(N=int(off[-1]), per_table=per_table, U=int(len(uk)), run_len=cnt, run_table=utab,
                hottest=int(cnt.max()) if len(cnt) else 0)


def byte_model(cfg, st, threshold=256, chunk=256, passes=None, bounds_ids=True, reuse_counts=False):
    """Algorithmic bytes of each stage for one step (what the method must move).  reuse_counts:
    the counts x table forward saves each bag's counts (128 bytes) and the backward reads them in
    place of the ids (ids past a bag's 256th, which it still reads, are left out of the model)."""
    wb = {"f32": 4, "f16": 2, "bf16": 2}[cfg.wdtype]
    ib = 4 if cfg.itype == "i32" else 8
    D = cfg.D.astype(np.int64)
    N, TB = st["N"], cfg.T * cfg.B
    pw = 4 if cfg.weighted else 0
    # tables served by the counts x table path (the library's eligibility rule)
    hist = np.array([t.histogram and cfg.wdtype == "f16" and not cfg.weighted and t.E <= 64 and 64 <= t.D <= 128
                     for t in cfg.tables])
    per_lookup = st["per_table"] * (D * wb + ib + pw)
    fwd = int(np.sum(per_lookup[~hist]) + int((~hist).sum()) * cfg.B * ib + cfg.B * int(D[~hist].sum()) * 4)
    counts_bytes = int(hist.sum()) * cfg.B * 128 if reuse_counts else 0
    hist_bytes = int(np.sum(st["per_table"][hist] * ib) + int(hist.sum()) * cfg.B * ib
                     + cfg.B * int(D[hist].sum()) * 4 + int(np.sum(cfg.E[hist] * D[hist] * wb)) + counts_bytes)
    hist_flops = int(np.sum(2 * cfg.B * cfg.E[hist] * D[hist]))
    # backward of those tables: counts^T x grad_out (ids and offsets again, the gradient slice,
    # the table and its state read and written once)
    ids_again = counts_bytes if reuse_counts else int(np.sum(st["per_table"][hist] * ib))
    bwd_hist = int(ids_again + int(hist.sum()) * cfg.B * ib
                   + cfg.B * int(D[hist].sum()) * 4 + int(np.sum(cfg.E[hist] * (2 * D[hist] * wb + 8))))
    bwd_hist_flops = hist_flops
    # gradient with respect to psw (weighted workloads): the rows again, the ids, one fp32 out per
    # lookup, each bag's gradient row once
    psw_grad = int(np.sum(st["per_table"] * (D * wb + ib + 4)) + TB * ib + cfg.B * int(D.sum()) * 4)
    bounds = (TB + 1) * ib + (N * ib if bounds_ids else 0)  # offsets (+ ids unless the forward checks them)
    # the sort only sees the other tables' lookups and runs
    N = N - int(np.sum(st["per_table"][hist]))
    run_keep = ~hist[st["run_table"]]
    if passes is None:  # the library's choice: digits of 8-10 bits, ceil(bits / 10) passes
        bits = 1
        while (1 << bits) <= cfg.total_rows:
            bits += 1
        passes = (bits + 9) // 10
    expand = N * (ib + 8 + 2 * pw) + TB * ib
    sort = passes * N * (20 + 2 * pw)
    U = int(run_keep.sum())
    rle = N * 8 + U * 8
    classify = U * 20
    Dr = D[st["run_table"][run_keep]]
    L = st["run_len"][run_keep]
    short = L < threshold
    upd_short = int(np.sum(L[short] * (4 + pw + Dr[short] * 4) + 2 * Dr[short] * wb + 8 + 16))
    nch = -(-L[~short] // chunk)
    upd_long = int(np.sum(L[~short] * (4 + pw + Dr[~short] * 4) + nch * Dr[~short] * 8
                          + 2 * Dr[~short] * wb + 8 + Dr[~short] * 4))
    n_hist = int(np.sum(st["per_table"][hist]))
    return dict(bounds=bounds, gather=fwd, histogram=hist_bytes, histogram_flops=hist_flops, expand=expand,
                sort=sort, rle=rle, classify=classify, short=upd_short, long=upd_long, apply=0,
                bwd_histogram=bwd_hist, bwd_histogram_flops=bwd_hist_flops, lookups_sorted=N, psw_grad=psw_grad,
                lookups_short=int(L[short].sum()), lookups_long=int(L[~short].sum()),
                lookups_gathered=st["N"] - n_hist, lookups_histogram=n_hist,
                runs_short=int(short.sum()), runs_long=int((~short).sum()), passes=passes)


# ------------------------------------------------------------------------------------------
# clocks during the timed region
# ------------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.tmp = None

    def start(self):
        self.tmp = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=self.tmp, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.tmp.flush()
        self.tmp.seek(0)
        rows = [r for r in csv.reader(io.StringIO(self.tmp.read())) if len(r) >= 9]
        self.tmp.close()
        os.unlink(self.tmp.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for name, v in zip(names, r[5:9]):
                if v.strip().lower().startswith("active"):
                    reasons.add(name)
        loaded = [s for s in sm if s > 0.5 * max(sm)] if sm else []
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------------------------------
# CPU oracle on a bounded sample of the workload
# ------------------------------------------------------------------------------------------
def oracle_sample(cfg, batch, bags_per_table: int):
    """The first `bags_per_table` bags of every table as a compact problem: each table keeps
    only the rows the sample touches, renamed to 0..k-1 in id order (so the grouping, the
    order of runs and every arithmetic step are those of the full problem on these bags),
    with the generator's values for those rows."""
    from synth.gen import grad_out_rows, weight_rows
    T, B = cfg.T, cfg.B
    S = min(bags_per_table, B)
    off = batch.offsets.astype(np.int64)
    new_off = [0]
    idx_parts, psw_parts, E_new, rows_per_table = [], [], [], []
    for t in range(T):
        s, e = off[t * B], off[t * B + S]
        ids = batch.indices[s:e].astype(np.int64)
        ok = (ids >= 0) & (ids < cfg.E[t])
        ids = np.where(ok, ids, 0)
        uniq, inv = np.unique(ids, return_inverse=True)
        if len(uniq) == 0:
            uniq = np.zeros(1, np.int64)
        idx_parts.append(inv.astype(np.int64))
        if batch.psw is not None:
            psw_parts.append(batch.psw[s:e])
        lens = np.diff(off[t * B:t * B + S + 1])
        new_off.extend((new_off[-1] + np.cumsum(lens)).tolist())
        E_new.append(len(uniq))
        rows_per_table.append(uniq)
    wd = cfg.wdtype
    parts = []
    for t in range(T):
        w = weight_rows(cfg, t, rows_per_table[t]).reshape(-1)
        parts.append(w.view(np.int16).numpy().view(np.uint16) if wd == "bf16" else w.numpy())
    weights = np.concatenate(parts)
    grad = grad_out_rows(cfg, np.arange(S)).numpy()
    return dict(T=T, B=S, D=cfg.D, E=np.array(E_new, np.int64), offsets=np.array(new_off, np.int64),
                indices=np.concatenate(idx_parts) if idx_parts else np.zeros(0, np.int64),
                psw=np.concatenate(psw_parts) if psw_parts else None, weights=weights, grad=grad,
                N=int(new_off[-1]))


def time_oracle(cfg, sample) -> tuple[float, float]:
    """Single-threaded oracle forward + backward on the sample; returns (seconds, lookups)."""
    import oracle
    tables = oracle.Tables(sample["D"], sample["E"])
    w = sample["weights"].copy()
    state = np.zeros(int(sample["E"].sum()), np.float32) if cfg.optimizer == "adagrad" else None
    t0 = time.perf_counter()
    oracle.forward(tables, sample["B"], w, sample["indices"], sample["offsets"], psw=sample["psw"], wdtype=cfg.wdtype)
    oracle.backward(tables, sample["B"], w, state, sample["indices"], sample["offsets"], sample["grad"],
                    psw=sample["psw"], optimizer=cfg.optimizer, lr=cfg.lr, eps=cfg.eps, wdtype=cfg.wdtype)
    return time.perf_counter() - t0, sample["N"]


def cpu_baseline(cfg, batch, bags: int, target_s: float = 15.0) -> dict:
    import oracle
    oracle.build()
    if bags <= 0:  # calibrate on a small sample, then size for ~target_s
        probe = oracle_sample(cfg, batch, max(1, min(cfg.B, 64)))
        dt, n = time_oracle(cfg, probe)
        rate = n / max(dt, 1e-6)
        mean_bag = max(1.0, batch.N / (cfg.T * cfg.B))
        bags = int(max(16, min(cfg.B, target_s * rate / (cfg.T * mean_bag))))
    sample = oracle_sample(cfg, batch, bags)
    dt, n = time_oracle(cfg, sample)
    return {"value": n / dt, "unit": "lookups/s", "cores": 1, "kind": "oracle",
            "seconds": round(dt, 3),
            "sample": f"first {sample['B']} of {cfg.B} bags of each of the {cfg.T} tables ({n} lookups), "
                      "rows renamed densely per table; forward + backward (one step), single thread; "
                      f"host has {os.cpu_count()} cores"}


# ------------------------------------------------------------------------------------------
# profile-derived DRAM traffic (valid only for the kernel source it was taken from)
# ------------------------------------------------------------------------------------------
def source_digest(files) -> str:
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


_CSRC = "bwd_tbe_fwd_gb300/csrc/"
KERNEL_SOURCES = {
    "gather": [_CSRC + "k_forward.cu", _CSRC + "tbe_internal.cuh"],
    # the update kernels walk the run lists in the classifier's order, which shapes their traffic
    "short": [_CSRC + "k_short.cu", _CSRC + "k_update_common.cuh", _CSRC + "k_classify.cu", _CSRC + "tbe_internal.cuh"],
    "long": [_CSRC + "k_long.cu", _CSRC + "k_update_common.cuh", _CSRC + "k_classify.cu", _CSRC + "tbe_internal.cuh"],
    "sort": [_CSRC + "k_sort.cu", _CSRC + "tbe_internal.cuh"],
    "histogram": [_CSRC + "k_hist.cu", _CSRC + "tbe_internal.cuh"],
    "bwd_histogram": [_CSRC + "k_hist.cu", _CSRC + "tbe_internal.cuh"],
}
# the lookups a stage's DRAM traffic is normalised by (ncu captures on smaller cases of the same
# workload, scaled to the full batch by these counts)
STAGE_UNITS = {"gather": "lookups_gathered", "short": "lookups_short", "long": "lookups_long",
               "sort": "lookups_sorted", "histogram": "lookups_histogram", "bwd_histogram": "lookups_histogram"}


def profiled_traffic(stage: str, workload: str, model: dict):
    """DRAM bytes (read + write) of one launch of the stage's kernel(s) on the full workload, from
    the ncu captures recorded in profiles/dram_traffic.json (bytes per lookup, scaled by the
    stage's lookups), with the capture's tensor-pipe utilisation if it has one; None when no
    capture exists or the kernel source changed since it was taken."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path) or stage not in KERNEL_SOURCES:
        return None
    with open(path) as f:
        table = json.load(f)
    rec = table.get(f"{workload}:{stage}")
    if not rec or rec.get("source_digest") != source_digest(KERNEL_SOURCES[stage]):
        return None
    units = model.get(STAGE_UNITS[stage], 0)
    if not units or "bytes_per_lookup" not in rec:
        return None
    return {"bytes": int(round(rec["bytes_per_lookup"] * units)), "from": rec.get("from"),
            "tensor_pipe_pct": rec.get("tensor_pipe_pct")}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


# ------------------------------------------------------------------------------------------
# our arm
# ------------------------------------------------------------------------------------------
class Workload:
    """One workload on the device: the batch, the library object, weights, state, gradients and
    the step of the hot path (bounds check, forward, backward update) through the C-ABI."""

    def __init__(self, args, cfg, dev, count_launches=False):
        import ctypes

        import torch
        from bwd_tbe_fwd_gb300 import TableBatchedEmbedding, TBEOptions
        from synth import make_batch
        from synth.gen import grad_out_tensor, torch_dtype, weights_tensor

        self.args, self.cfg, self.dev = args, cfg, dev
        self.batch = make_batch(cfg)
        self.st = batch_stats(cfg, self.batch)
        self.opts = TBEOptions(long_mode={"auto": 0, "two_kernel": 1, "fused": 2}[args.long_mode],
                               scheduler={"grid": 0, "persistent": 1, "clc": 2}[args.scheduler],
                               merge={"atomic": 0, "bulk": 1}[args.merge],
                               gather={"register": 0, "tma": 1}[args.gather],
                               fused_bounds=1 if args.bounds == "fused" else 0,
                               classify_mode={"atomic": 0, "ordered": 1}[args.classify])
        itype = torch.int32 if cfg.itype == "i32" else torch.int64
        self.tbe = TableBatchedEmbedding(cfg.D, cfg.E, cfg.B, self.batch.N, torch_dtype(cfg.wdtype), itype,
                                         weighted=cfg.weighted, long_bags=[t.histogram for t in cfg.tables],
                                         device=dev, options=self.opts, pooling=args.pooling)
        self.psw_grad = args.psw_grad and cfg.weighted
        self.grad_psw = torch.empty(self.batch.N, dtype=torch.float32, device=dev) if self.psw_grad else None
        self.weights = weights_tensor(cfg, device=dev)
        self.state = (torch.zeros(cfg.total_rows, dtype=torch.float32, device=dev)
                      if cfg.optimizer == "adagrad" else None)
        self.grad = grad_out_tensor(cfg, device=dev)
        self.idx_h = torch.from_numpy(self.batch.indices)
        self.off_h = torch.from_numpy(self.batch.offsets)
        self.psw_h = None if self.batch.psw is None else torch.from_numpy(self.batch.psw)
        self.inputs = (self.idx_h.to(dev), self.off_h.to(dev), None if self.psw_h is None else self.psw_h.to(dev))
        self.out = torch.empty(cfg.B, cfg.total_D, dtype=torch.float32, device=dev)
        self.stats = torch.zeros(8, dtype=torch.int64, device=dev)
        self.launches = ctypes.c_int64(0)
        if count_launches:
            self.opts.count_launches(self.launches)
        self.main = torch.cuda.current_stream(dev)
        self.side = torch.cuda.Stream(device=dev, priority=-1)  # its CTAs go first when SMs free up
        self.model = byte_model(cfg, self.st, self.opts.c.long_threshold, self.opts.c.chunk,
                                bounds_ids=args.bounds != "fused", reuse_counts=args.reuse_counts == "on")

    def step(self, fev=None, bev=None, bounds_ev=None, pev=None, gev=None, ins=None):
        args, tbe, cfg = self.args, self.tbe, self.cfg
        idx, off, psw = ins if ins is not None else self.inputs
        if bounds_ev is not None:
            bounds_ev[0].record()
        tbe.bounds_check(idx, off, stats=self.stats, offsets_only=args.bounds == "fused")
        if bounds_ev is not None:
            bounds_ev[1].record()
        if args.hoist == "on":
            # the transpose needs only the repaired ids: run it beside the forward gather
            self.side.wait_stream(self.main)
            self.opts.with_events(pev)
            tbe.backward_prepare(idx, off, psw=psw, stats=self.stats, stream=self.side)
        self.opts.with_events(fev)
        tbe.forward(self.weights, idx, off, psw=psw, out=self.out, stats=self.stats)
        if args.hoist == "on":
            self.main.wait_stream(self.side)
        if self.psw_grad:
            if gev is not None:
                gev[0].record()
            tbe.psw_gradient(self.weights, idx, off, self.grad, grad_psw=self.grad_psw)
            if gev is not None:
                gev[1].record()
        self.opts.with_events(bev)
        tbe.backward_update(self.weights, self.state, idx, off, self.grad, psw=psw, optimizer=cfg.optimizer,
                            lr=cfg.lr, eps=cfg.eps, stats=self.stats, prepared=args.hoist == "on",
                            reuse_forward=args.reuse_counts == "on")
        self.opts.with_events(None)

    def timed(self, K, W, world=1, clocks=None):
        """W untimed steps, then K timed ones (CUDA events on the launching stream, barrier and
        synchronize on both sides); per-stage device times from the library's stage events."""
        import torch
        from bwd_tbe_fwd_gb300.tbe import BWD_STAGES, TBE_BWD_NUM_EVENTS, TBE_FWD_NUM_EVENTS
        for _ in range(W):
            self.step()
        torch.cuda.synchronize()
        mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
        fevs = [[mk() for _ in range(TBE_FWD_NUM_EVENTS)] for _ in range(K)]
        bevs = [[mk() for _ in range(TBE_BWD_NUM_EVENTS)] for _ in range(K)]
        bnds = [[mk(), mk()] for _ in range(K)]
        pevs = [[mk() for _ in range(TBE_BWD_NUM_EVENTS)] for _ in range(K)]
        gevs = [[mk(), mk()] for _ in range(K)]
        e0, e1 = mk(), mk()
        hoist = self.args.hoist == "on"
        self.launches.value = 0
        barrier(world)
        torch.cuda.synchronize()
        if clocks is not None:
            clocks.start()
            time.sleep(0.4)  # let the sampler take a first sample
        e0.record()
        for k in range(K):
            self.step(fevs[k], bevs[k], bnds[k], pevs[k] if hoist else None, gevs[k])
        e1.record()
        torch.cuda.synchronize()
        clk = clocks.stop() if clocks is not None else None
        barrier(world)
        stage_ms = {"bounds": np.mean([b[0].elapsed_time(b[1]) for b in bnds]),
                    "psw_grad": np.mean([g[0].elapsed_time(g[1]) for g in gevs]) if self.psw_grad else 0.0,
                    "gather": np.mean([f[0].elapsed_time(f[1]) for f in fevs]),
                    "histogram": np.mean([f[1].elapsed_time(f[2]) for f in fevs])}
        for i, name in enumerate(BWD_STAGES):
            # with the transpose hoisted, its stages ran on the side stream between the prepare's events
            src = pevs if hoist and name in ("expand", "sort", "rle", "classify") else bevs
            stage_ms[name] = float(np.mean([b[i].elapsed_time(b[i + 1]) for b in src]))
        return {"ms_total": e0.elapsed_time(e1), "stage_ms": stage_ms, "clocks": clk,
                "launches": int(self.launches.value),
                "fwd_ms": float(np.mean([f[0].elapsed_time(f[2]) for f in fevs])),
                "bwd_ms": float(np.mean([b[0].elapsed_time(b[-1]) for b in bevs]))}

    def roofline(self, stage_ms, peak, peak_kind):
        """Per-stage algorithmic bytes and, where an ncu capture of the current kernel source exists,
        DRAM bytes; the roofline of the slowest kernel stage against the HBM copy peak, by DRAM bytes.
        Algorithmic bytes count every row read, most of which the skewed ids make L2 hits, so their
        rate is an L2-served figure, not a fraction of HBM."""
        model, cfg = self.model, self.cfg
        stages = {}
        for name, ms in stage_ms.items():
            gb = model.get(name, 0) / 1e9
            rec = {"ms": round(float(ms), 4), "algorithmic_GB": round(gb, 4),
                   "algorithmic_GBps": round(gb / (ms / 1e3), 1) if ms > 0 and gb > 0 else None}
            tr = profiled_traffic(name, cfg.name, model) if ms > 0 else None
            if tr is not None:
                rec["dram_GB"] = round(tr["bytes"] / 1e9, 4)
                rec["dram_GBps"] = round(tr["bytes"] / 1e9 / (ms / 1e3), 1)
                rec["dram_frac"] = round(tr["bytes"] / 1e9 / (ms / 1e3) / peak, 4)
                if tr.get("tensor_pipe_pct") is not None:
                    rec["tensor_pipe_pct"] = tr["tensor_pipe_pct"]
            stages[name] = rec
        for name in ("histogram", "bwd_histogram"):
            if model[name + "_flops"] > 0 and stage_ms[name] > 0:
                stages[name]["tensor_TFLOPs"] = round(model[name + "_flops"] / (stage_ms[name] / 1e3) / 1e12, 3)
        kernel_stages = ("gather", "histogram", "short", "long", "bwd_histogram")
        dom = max(kernel_stages, key=lambda n: stage_ms[n])
        tr = profiled_traffic(dom, cfg.name, model)
        ms = stage_ms[dom]
        achieved = tr["bytes"] / 1e9 / (ms / 1e3) if tr is not None else None
        roof = {"kernel": dom, "bound": "hbm", "achieved": round(achieved, 1) if achieved is not None else None,
                "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                "frac": round(achieved / peak, 4) if achieved is not None else None,
                "traffic": tr["bytes"] if tr is not None else None,
                "traffic_from": tr["from"] if tr is not None else None,
                "algorithmic_bytes": model[dom],
                "algorithmic_GBps": round(model[dom] / 1e9 / (ms / 1e3), 1),
                "basis": "achieved = ncu DRAM bytes (read + write) of the kernel per launch, from a capture of "
                         "the current kernel source scaled to this batch by its lookups, over the kernel's CUDA-event "
                         "time; algorithmic_GBps counts every row read (mostly L2 hits) and is not an HBM fraction"}
        return stages, roof

    def release(self):
        import torch
        for k in ("tbe", "weights", "state", "grad", "inputs", "out", "stats", "grad_psw"):
            setattr(self, k, None)
        torch.cuda.empty_cache()


def per_config_lines(args, dev, K, W, peak, peak_kind):
    """The other workloads, each timed in this process after the headline one."""
    from synth import get_config
    res = {}
    for name in args.per_config.split(","):
        name = name.strip()
        if not name or name == args.config:
            continue
        cfg = get_config(name)
        wl = Workload(args, cfg, dev)
        t = wl.timed(K, W)
        stages, roof = wl.roofline(t["stage_ms"], peak, peak_kind)
        line = {"workload": f"{cfg.name}: {cfg.description}", "lookups_per_step": wl.st["N"],
                "ms_per_step": round(t["ms_total"] / K, 4),
                "value": wl.st["N"] * K / (t["ms_total"] / 1e3), "unit": "lookups/s",
                "fwd_ms": round(t["fwd_ms"], 4), "bwd_ms": round(t["bwd_ms"], 4), "steps": K, "warmup": W,
                "roofline": roof,
                "dram_frac": {n: stages[n].get("dram_frac") for n in ("gather", "short", "long", "histogram",
                                                                     "bwd_histogram") if stages[n]["ms"] > 0.003},
                "stages": stages}
        res[cfg.name] = line
        wl.release()
        del wl
    return res


def run_ours(args):
    import torch
    from bwd_tbe_fwd_gb300 import build
    from synth import get_config

    world, rank, local = dist_setup("nccl")
    build.build()
    dev = torch.device("cuda", local)
    cfg = get_config(args.config)
    if args.tables:
        cfg = cfg.shrink(T=args.tables, name=f"{cfg.name}[T={args.tables}]")
    if args.bags:
        cfg = cfg.shrink(B=args.bags, name=f"{cfg.name}[B={args.bags}]")
    wl = Workload(args, cfg, dev, count_launches=True)
    st, model = wl.st, wl.model
    K = args.steps
    clocks = ClockSampler(local)
    t = wl.timed(K, args.warmup, world, clocks)
    clk = t["clocks"]
    gpu_launches = t["launches"] + K * BOUNDS_LAUNCHES[args.bounds]
    ms_total = t["ms_total"]
    ms_max = all_max(world, ms_total, dev)
    lookups_all = all_sum(world, float(st["N"]) * K, dev)
    peak, peak_kind = peaks()
    stages, roof = wl.roofline(t["stage_ms"], peak, peak_kind)

    # end to end: host inputs copied in, the step, the step's counters read back
    e2e = None
    if not args.no_e2e:
        idx_p = wl.idx_h.pin_memory()
        off_p = wl.off_h.pin_memory()
        psw_p = None if wl.psw_h is None else wl.psw_h.pin_memory()
        stats_p = torch.zeros(8, dtype=torch.int64).pin_memory()
        h2d = idx_p.numel() * idx_p.element_size() + off_p.numel() * off_p.element_size()
        if psw_p is not None:
            h2d += psw_p.numel() * 4
        # Two device copies of the inputs: step k's copy (on a copy stream) overlaps step k-1's
        # work; a step starts when its inputs have landed, a buffer is refilled once the step
        # that used it is done.
        idx, off, psw = wl.inputs
        bufs = [wl.inputs, (torch.empty_like(idx), torch.empty_like(off), None if psw is None else torch.empty_like(psw))]
        copy = torch.cuda.Stream(device=dev)
        landed = [torch.cuda.Event(), torch.cuda.Event()]
        used = [torch.cuda.Event(), torch.cuda.Event()]

        def upload(k):
            b = bufs[k % 2]
            with torch.cuda.stream(copy):
                if k >= 2:
                    copy.wait_event(used[k % 2])
                b[0].copy_(idx_p, non_blocking=True)
                b[1].copy_(off_p, non_blocking=True)
                if psw_p is not None:
                    b[2].copy_(psw_p, non_blocking=True)
                landed[k % 2].record(copy)

        torch.cuda.synchronize()
        barrier(world)
        t0 = time.perf_counter()
        upload(0)
        for k in range(K):
            if k + 1 < K:
                upload(k + 1)
            wl.main.wait_event(landed[k % 2])
            wl.step(ins=bufs[k % 2])
            used[k % 2].record(wl.main)
            stats_p.copy_(wl.stats, non_blocking=True)
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
        dt = all_max(world, dt, dev)
        e2e = {"value": lookups_all / dt, "unit": "lookups/s", "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": 64, "ms_per_step": round(dt * 1e3 / K, 3),
               "note": "per step: indices+offsets (+psw) pinned host->device (on a copy stream, double "
                       "buffered: step k+1's copy overlaps step k), bounds+forward+backward, the step's "
                       "int64 counters device->host; wall clock over all steps"}

    # the other classifier on the same workload: [FBT] section 4, Problem 4 names one atomic per
    # block per list (ATOMIC); ORDERED writes the lists in key order (the default)
    side = None
    if rank == 0 and world == 1 and not args.no_side:
        from bwd_tbe_fwd_gb300.tbe import TBE_CLASSIFY_ATOMIC, TBE_CLASSIFY_ORDERED
        keep = wl.opts.c.classify_mode
        wl.opts.c.classify_mode = TBE_CLASSIFY_ATOMIC if keep == TBE_CLASSIFY_ORDERED else TBE_CLASSIFY_ORDERED
        ks = min(K, 10)
        ts = wl.timed(ks, 3)
        wl.opts.c.classify_mode = keep
        side = {"classify": "atomic" if keep == TBE_CLASSIFY_ORDERED else "ordered", "steps": ks,
                "ms_per_step": round(ts["ms_total"] / ks, 4),
                "stages_ms": {k: round(float(ts["stage_ms"][k]), 4) for k in ("classify", "short", "long")}}
    # the transpose hoisted beside the forward ([FBT] section 3: the backward's metadata built
    # while the forward runs): a few steps with --hoist flipped; the stage times then overlap, so
    # the headline and its roofline stay on the sequential step
    hoisted = None
    if rank == 0 and world == 1 and not args.no_side:
        keep_h = wl.args.hoist
        wl.args.hoist = "on" if keep_h == "off" else "off"
        ks = min(K, 10)
        th = wl.timed(ks, 3)
        hoisted = {"hoist": wl.args.hoist, "steps": ks, "ms_per_step": round(th["ms_total"] / ks, 4),
                   "value": float(st["N"]) / (th["ms_total"] / ks / 1e3),
                   "stages_ms": {k: round(float(th["stage_ms"][k]), 4) for k in ("gather", "expand", "sort", "short", "long")},
                   "note": "overlapped stages: gather and the transpose share the SMs"}
        wl.args.hoist = keep_h

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(cfg, wl.batch, args.cpu_sample_bags)
    batch_desc = {"lookups_per_step": st["N"], "distinct_rows": st["U"], "hottest_row_hits": st["hottest"],
                  "long_runs": model["runs_long"], "lookups_in_long_runs": model["lookups_long"]}
    wl.release()

    per_config = None
    if rank == 0 and world == 1 and args.per_config:
        per_config = per_config_lines(args, dev, min(K, 20), max(3, min(args.warmup, 5)), peak, peak_kind)

    if rank == 0:
        line = {
            "metric": METRIC,
            "value": lookups_all / (ms_max / 1e3),
            "unit": "lookups/s",
            "n_gpus": world,
            "steps": K,
            "warmup": args.warmup,
            "ms_per_step": round(ms_max / K, 4),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "f32",
            "data": "synthetic",
            "config": {
                "workload": f"{cfg.name}: {cfg.description}",
                **batch_desc,
                "weights_storage": cfg.wdtype, "step": (("tbe_bounds_check_offsets" if args.bounds == "fused" else "tbe_bounds_check")
                         + (" + (tbe_forward || tbe_backward_prepare) + tbe_backward_update(prepared)"
                            if args.hoist == "on" else " + tbe_forward + tbe_backward_update")
                         + (" (ids repaired inside tbe_forward)" if args.bounds == "fused" else "")),
                "long_mode": args.long_mode, "scheduler": args.scheduler, "merge": args.merge, "gather": args.gather, "classify": args.classify,
                "transpose": "hoisted beside the forward (second stream)" if args.hoist == "on" else "in the backward",
                "counts_reuse": args.reuse_counts == "on",
                "pooling": args.pooling, "psw_grad": bool(wl.psw_grad),
                "parallelism": f"replicas x{world}",
                "l2": "inputs larger than L2 (weights alone exceed 129 MB); no flush between steps",
                "fwd_ms": round(t["fwd_ms"], 4), "bwd_ms": round(t["bwd_ms"], 4),
            },
            "roofline": roof,
            "stages": stages,
            "per_config": per_config,
            "classify_alternative": side,
            "hoist_alternative": hoisted,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "clocks": clk,
            "gpu_launches": gpu_launches,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ------------------------------------------------------------------------------------------
# reference arm: the CPU oracle on bounded samples of the same workload
# ------------------------------------------------------------------------------------------
def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from synth import get_config, make_batch
    import oracle
    oracle.build()
    cfg = get_config(args.config)
    batch = make_batch(cfg)
    # size each step for ~4 s so that warmup + steps end within a few minutes
    probe = oracle_sample(cfg, batch, 32)
    dt, n = time_oracle(cfg, probe)
    rate = n / max(dt, 1e-6)
    total_steps = args.steps + args.warmup
    per_step_s = max(0.5, min(4.0, 150.0 / max(1, total_steps)))
    bags = int(max(8, min(cfg.B, per_step_s * rate / max(1.0, batch.N / cfg.B))))
    sample = oracle_sample(cfg, batch, bags)
    for _ in range(args.warmup):
        time_oracle(cfg, sample)
    times = [time_oracle(cfg, sample)[0] for _ in range(args.steps)]
    total = float(np.sum(times))
    value = sample["N"] * args.steps / total
    desc = (f"first {sample['B']} of {cfg.B} bags of each of the {cfg.T} tables ({sample['N']} lookups) "
            "per step, rows renamed densely per table; oracle forward + backward, single thread")
    line = {
        "metric": METRIC, "value": value, "unit": "lookups/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total * 1e3 / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
        "config": {"workload": f"{cfg.name}: {cfg.description}", "sample": desc},
        "cpu_baseline": {"value": value, "unit": "lookups/s", "cores": 1, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "lookups/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
