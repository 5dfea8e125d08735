"""Host-side logic of bench.py on the CPU: the byte model, the workload statistics, the
reference arm's JSON line, and the multi-process (replicas) helpers on a world of two gloo ranks."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import oracle  # noqa: E402
from synth import get_config, make_batch  # noqa: E402


def test_batch_stats_match_the_oracle_runs():
    cfg = get_config("c2").shrink(B=256, E_div=1000)
    batch = make_batch(cfg)
    st = bench.batch_stats(cfg, batch)
    idx, off = batch.indices.copy(), batch.offsets.copy()
    oracle.bounds_repair(oracle.Tables(cfg.D, cfg.E), cfg.B, idx, off)
    w = np.zeros(int((cfg.E * cfg.D).sum()), dtype=np.float16)
    res = oracle.backward(oracle.Tables(cfg.D, cfg.E), cfg.B, w, None, idx, off,
                          np.zeros((cfg.B, int(cfg.D.sum())), np.float32), optimizer="sgd")
    assert st["N"] == res["num_lookups"] and st["U"] == res["num_runs"]
    assert np.array_equal(np.sort(st["run_len"]), np.sort(res["run_lengths"]))


def test_byte_model_counts_and_histogram_split():
    cfg = get_config("c4").shrink(B=512, E_div=100)
    batch = make_batch(cfg)
    st = bench.batch_stats(cfg, batch)
    m = bench.byte_model(cfg, st)
    # table 0 is on the counts path: its lookups skip the sort, the long path and the gather
    n0 = int(st["per_table"][0])
    assert m["lookups_sorted"] == st["N"] - n0
    assert m["histogram"] > 0 and m["bwd_histogram"] > 0 and m["histogram_flops"] == 2 * cfg.B * 64 * 128
    assert m["lookups_short"] + m["lookups_long"] == st["N"] - n0
    # forward bytes of the gathered table: rows, ids, offsets and output
    ib, D1 = 8, int(cfg.D[1])
    assert m["gather"] == int(st["per_table"][1]) * (D1 * 2 + ib) + cfg.B * ib + cfg.B * D1 * 4
    for k in ("expand", "sort", "rle", "classify", "short", "psw_grad", "bounds"):
        assert m[k] >= 0


def test_byte_model_with_the_forward_counts_reused():
    """With the forward's counts reused, the counts-path forward also writes 128 bytes per bag
    and the backward reads those instead of the table's ids; nothing else changes."""
    cfg = get_config("c4").shrink(B=512, E_div=100)
    st = bench.batch_stats(cfg, make_batch(cfg))
    m0 = bench.byte_model(cfg, st)
    m1 = bench.byte_model(cfg, st, reuse_counts=True)
    ids0 = int(st["per_table"][0]) * 8
    assert m1["histogram"] - m0["histogram"] == cfg.B * 128
    assert m0["bwd_histogram"] - m1["bwd_histogram"] == ids0 - cfg.B * 128
    for k in ("gather", "expand", "sort", "rle", "classify", "short", "long", "lookups_histogram"):
        assert m0[k] == m1[k], k


def test_reference_arm_prints_one_line():
    env = dict(os.environ, PYTHONPATH=ROOT)
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "c1",
                          "--steps", "2", "--warmup", "1"], capture_output=True, text=True, env=env, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["value"] > 0 and d["steps"] == 2
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"


def test_reference_arm_other_ranks_print_nothing():
    env = dict(os.environ, PYTHONPATH=ROOT, RANK="1", WORLD_SIZE="2")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "c1",
                          "--steps", "1", "--warmup", "0"], capture_output=True, text=True, env=env, timeout=600)
    assert out.returncode == 0 and out.stdout.strip() == ""


_WORKER = r"""
import os, sys, json
sys.path.insert(0, {root!r})
import bench
world, rank, local = bench.dist_setup("gloo")
bench.barrier(world)
mx = bench.all_max(world, 1.5 + rank, "cpu")
sm = bench.all_sum(world, 10.0 * (rank + 1), "cpu")
bench.barrier(world)
print(json.dumps({{"rank": rank, "world": world, "max": mx, "sum": sm}}))
import torch.distributed as dist
dist.destroy_process_group()
"""


def test_replica_reductions_on_two_gloo_ranks(tmp_path):
    """The N>1 bench path: each replica times its own batch; the line reports all ranks'
    lookups over the slowest rank's time (max and sum across two gloo ranks)."""
    script = tmp_path / "worker.py"
    script.write_text(_WORKER.format(root=ROOT))
    procs = []
    for r in range(2):
        env = dict(os.environ, RANK=str(r), LOCAL_RANK=str(r), WORLD_SIZE="2", MASTER_ADDR="127.0.0.1",
                   MASTER_PORT="29517")
        procs.append(subprocess.Popen([sys.executable, str(script)], stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True, env=env))
    outs = [p.communicate(timeout=300) for p in procs]
    for p, (o, e) in zip(procs, outs):
        assert p.returncode == 0, e[-2000:]
    res = sorted((json.loads(o.strip().splitlines()[-1]) for o, _ in outs), key=lambda d: d["rank"])
    assert [d["rank"] for d in res] == [0, 1] and all(d["world"] == 2 for d in res)
    assert all(d["max"] == 2.5 and d["sum"] == 30.0 for d in res)
