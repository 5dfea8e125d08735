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
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--tables", type=int, default=0,
                    help="keep only the first T tables of the workload (small cases for profiling)")
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


def byte_model(cfg, st, threshold=256, chunk=256, passes=None, bounds_ids=True):
    """Algorithmic bytes of each stage for one step (what the method must move)."""
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
    hist_bytes = int(np.sum(st["per_table"][hist] * ib) + int(hist.sum()) * cfg.B * ib
                     + cfg.B * int(D[hist].sum()) * 4 + int(np.sum(cfg.E[hist] * D[hist] * wb)))
    hist_flops = int(np.sum(2 * cfg.B * cfg.E[hist] * D[hist]))
    # backward of those tables: counts^T x grad_out (ids and offsets again, the gradient slice,
    # the table and its state read and written once)
    bwd_hist = int(np.sum(st["per_table"][hist] * ib) + int(hist.sum()) * cfg.B * ib
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
    return dict(bounds=bounds, gather=fwd, histogram=hist_bytes, histogram_flops=hist_flops, expand=expand,
                sort=sort, rle=rle, classify=classify, short=upd_short, long=upd_long, apply=0,
                bwd_histogram=bwd_hist, bwd_histogram_flops=bwd_hist_flops, lookups_sorted=N, psw_grad=psw_grad,
                lookups_short=int(L[short].sum()), lookups_long=int(L[~short].sum()),
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
    "short": [_CSRC + "k_short.cu", _CSRC + "k_update_common.cuh", _CSRC + "tbe_internal.cuh"],
    "long": [_CSRC + "k_long.cu", _CSRC + "k_update_common.cuh", _CSRC + "tbe_internal.cuh"],
    "sort": [_CSRC + "k_sort.cu", _CSRC + "tbe_internal.cuh"],
    "histogram": [_CSRC + "k_hist.cu", _CSRC + "tbe_internal.cuh"],
    "bwd_histogram": [_CSRC + "k_hist.cu", _CSRC + "tbe_internal.cuh"],
}


def profiled_traffic(stage: str, workload: str):
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(path) or stage not in KERNEL_SOURCES:
        return None
    with open(path) as f:
        table = json.load(f)
    rec = table.get(f"{workload}:{stage}")
    if not rec or rec.get("source_digest") != source_digest(KERNEL_SOURCES[stage]):
        return None
    return rec.get("bytes_per_launch")


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
def run_ours(args):
    import ctypes

    import torch
    from bwd_tbe_fwd_gb300 import TableBatchedEmbedding, TBEOptions, build
    from bwd_tbe_fwd_gb300.tbe import BWD_STAGES, TBE_BWD_NUM_EVENTS, TBE_FWD_NUM_EVENTS
    from synth import get_config, make_batch
    from synth.gen import grad_out_tensor, torch_dtype, weights_tensor

    world, rank, local = dist_setup("nccl")
    build.build()
    dev = torch.device("cuda", local)
    cfg = get_config(args.config)
    if args.tables:
        cfg = cfg.shrink(T=args.tables, name=f"{cfg.name}[T={args.tables}]")
    batch = make_batch(cfg)
    st = batch_stats(cfg, batch)
    opts = TBEOptions(long_mode={"auto": 0, "two_kernel": 1, "fused": 2}[args.long_mode],
                      scheduler={"grid": 0, "persistent": 1, "clc": 2}[args.scheduler],
                      merge={"atomic": 0, "bulk": 1}[args.merge],
                      gather={"register": 0, "tma": 1}[args.gather],
                      fused_bounds=1 if args.bounds == "fused" else 0,
                      classify_mode={"atomic": 0, "ordered": 1}[args.classify])
    itype = torch.int32 if cfg.itype == "i32" else torch.int64
    tbe = TableBatchedEmbedding(cfg.D, cfg.E, cfg.B, batch.N, torch_dtype(cfg.wdtype), itype,
                                weighted=cfg.weighted, long_bags=[t.histogram for t in cfg.tables],
                                device=dev, options=opts, pooling=args.pooling)
    psw_grad = args.psw_grad and cfg.weighted
    grad_psw = torch.empty(batch.N, dtype=torch.float32, device=dev) if psw_grad else None
    weights = weights_tensor(cfg, device=dev)
    state = torch.zeros(cfg.total_rows, dtype=torch.float32, device=dev) if cfg.optimizer == "adagrad" else None
    grad = grad_out_tensor(cfg, device=dev)
    idx_h = torch.from_numpy(batch.indices)
    off_h = torch.from_numpy(batch.offsets)
    psw_h = None if batch.psw is None else torch.from_numpy(batch.psw)
    idx = idx_h.to(dev)
    off = off_h.to(dev)
    psw = None if psw_h is None else psw_h.to(dev)
    out = torch.empty(cfg.B, cfg.total_D, dtype=torch.float32, device=dev)
    stats = torch.zeros(8, dtype=torch.int64, device=dev)
    launches = ctypes.c_int64(0)
    opts.count_launches(launches)

    main = torch.cuda.current_stream(dev)
    side = torch.cuda.Stream(device=dev, priority=-1)  # its CTAs go first when SMs free up
    inputs = (idx, off, psw)

    def step(fev=None, bev=None, bounds_ev=None, pev=None, gev=None, ins=None):
        idx, off, psw = ins if ins is not None else inputs
        if bounds_ev is not None:
            bounds_ev[0].record()
        tbe.bounds_check(idx, off, stats=stats, offsets_only=args.bounds == "fused")
        if bounds_ev is not None:
            bounds_ev[1].record()
        if args.hoist == "on":
            # the transpose needs only the repaired ids: run it beside the forward gather
            side.wait_stream(main)
            opts.with_events(pev)
            tbe.backward_prepare(idx, off, psw=psw, stats=stats, stream=side)
        opts.with_events(fev)
        tbe.forward(weights, idx, off, psw=psw, out=out, stats=stats)
        if args.hoist == "on":
            main.wait_stream(side)
        if psw_grad:
            if gev is not None:
                gev[0].record()
            tbe.psw_gradient(weights, idx, off, grad, grad_psw=grad_psw)
            if gev is not None:
                gev[1].record()
        opts.with_events(bev)
        tbe.backward_update(weights, state, idx, off, grad, psw=psw, optimizer=cfg.optimizer, lr=cfg.lr,
                            eps=cfg.eps, stats=stats, prepared=args.hoist == "on")
        opts.with_events(None)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    K = args.steps
    mk = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    fevs = [[mk() for _ in range(TBE_FWD_NUM_EVENTS)] for _ in range(K)]
    bevs = [[mk() for _ in range(TBE_BWD_NUM_EVENTS)] for _ in range(K)]
    bnds = [[mk(), mk()] for _ in range(K)]
    pevs = [[mk() for _ in range(TBE_BWD_NUM_EVENTS)] for _ in range(K)]
    gevs = [[mk(), mk()] for _ in range(K)]
    e0, e1 = mk(), mk()
    clocks = ClockSampler(local)
    launches.value = 0
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.4)  # let the sampler take a first sample
    e0.record()
    for k in range(K):
        step(fevs[k], bevs[k], bnds[k], pevs[k] if args.hoist == "on" else None, gevs[k])
    e1.record()
    torch.cuda.synchronize()
    clk = clocks.stop()
    barrier(world)
    gpu_launches = int(launches.value) + K * BOUNDS_LAUNCHES[args.bounds]
    ms_total = e0.elapsed_time(e1)
    ms_max = all_max(world, ms_total, dev)
    lookups_all = all_sum(world, float(st["N"]) * K, dev)

    # per-stage device times (ms per step)
    stage_ms = {"bounds": np.mean([b[0].elapsed_time(b[1]) for b in bnds]),
                "psw_grad": np.mean([g[0].elapsed_time(g[1]) for g in gevs]) if psw_grad else 0.0,
                "gather": np.mean([f[0].elapsed_time(f[1]) for f in fevs]),
                "histogram": np.mean([f[1].elapsed_time(f[2]) for f in fevs])}
    for i, name in enumerate(BWD_STAGES):
        # with the transpose hoisted, its stages ran on the side stream between the prepare's events
        src = pevs if args.hoist == "on" and name in ("expand", "sort", "rle", "classify") else bevs
        stage_ms[name] = float(np.mean([b[i].elapsed_time(b[i + 1]) for b in src]))
    fwd_ms = float(np.mean([f[0].elapsed_time(f[2]) for f in fevs]))
    bwd_ms = float(np.mean([b[0].elapsed_time(b[-1]) for b in bevs]))
    model = byte_model(cfg, st, opts.c.long_threshold, opts.c.chunk, bounds_ids=args.bounds != "fused")
    peak, peak_kind = peaks()
    stages = {}
    for name, ms in stage_ms.items():
        gb = model.get(name, 0) / 1e9
        stages[name] = {"ms": round(float(ms), 4), "algorithmic_GB": round(gb, 4),
                        "GBps": round(gb / (ms / 1e3), 1) if ms > 0 and gb > 0 else None,
                        "frac": round(gb / (ms / 1e3) / peak, 4) if ms > 0 and gb > 0 else None}
    for name in ("histogram", "bwd_histogram"):
        if model[name + "_flops"] > 0 and stage_ms[name] > 0:
            stages[name]["tensor_TFLOPs"] = round(model[name + "_flops"] / (stage_ms[name] / 1e3) / 1e12, 3)
    kernel_stages = ("gather", "histogram", "short", "long", "bwd_histogram")
    dom = max(kernel_stages, key=lambda n: stage_ms[n])
    achieved = model[dom] / 1e9 / (stage_ms[dom] / 1e3)
    traffic = profiled_traffic(dom, cfg.name)

    # end to end: host inputs copied in, the step, the step's counters read back
    e2e = None
    if not args.no_e2e:
        idx_p = idx_h.pin_memory()
        off_p = off_h.pin_memory()
        psw_p = None if psw_h is None else psw_h.pin_memory()
        stats_p = torch.zeros(8, dtype=torch.int64).pin_memory()
        h2d = idx_p.numel() * idx_p.element_size() + off_p.numel() * off_p.element_size()
        if psw_p is not None:
            h2d += psw_p.numel() * 4
        # Two device copies of the inputs: step k's copy (on a copy stream) overlaps step k-1's
        # work; a step starts when its inputs have landed, a buffer is refilled once the step
        # that used it is done.
        bufs = [inputs, (torch.empty_like(idx), torch.empty_like(off), None if psw is None else torch.empty_like(psw))]
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
            main.wait_event(landed[k % 2])
            step(ins=bufs[k % 2])
            used[k % 2].record(main)
            stats_p.copy_(stats, non_blocking=True)
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
        dt = all_max(world, dt, dev)
        e2e = {"value": lookups_all / dt, "unit": "lookups/s", "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": 64, "ms_per_step": round(dt * 1e3 / K, 3),
               "note": "per step: indices+offsets (+psw) pinned host->device (on a copy stream, double "
                       "buffered: step k+1's copy overlaps step k), bounds+forward+backward, the step's "
                       "int64 counters device->host; wall clock over all steps"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(cfg, batch, args.cpu_sample_bags)

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
                "lookups_per_step": st["N"], "distinct_rows": st["U"], "hottest_row_hits": st["hottest"],
                "long_runs": model["runs_long"], "lookups_in_long_runs": model["lookups_long"],
                "weights_storage": cfg.wdtype, "step": (("tbe_bounds_check_offsets" if args.bounds == "fused" else "tbe_bounds_check")
                         + (" + (tbe_forward || tbe_backward_prepare) + tbe_backward_update(prepared)"
                            if args.hoist == "on" else " + tbe_forward + tbe_backward_update")
                         + (" (ids repaired inside tbe_forward)" if args.bounds == "fused" else "")),
                "long_mode": args.long_mode, "scheduler": args.scheduler, "merge": args.merge, "gather": args.gather, "classify": args.classify,
                "transpose": "hoisted beside the forward (second stream)" if args.hoist == "on" else "in the backward",
                "pooling": args.pooling, "psw_grad": bool(psw_grad),
                "parallelism": f"replicas x{world}",
                "l2": "inputs larger than L2 (weights alone exceed 129 MB); no flush between steps",
                "fwd_ms": round(fwd_ms, 4), "bwd_ms": round(bwd_ms, 4),
            },
            "roofline": {"kernel": dom, "bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                         "peak_kind": peak_kind, "unit": "GB/s", "frac": round(achieved / peak, 4),
                         "traffic": traffic, "algorithmic_bytes": model[dom]},
            "stages": stages,
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
