"""tbe_backward_update_noalloc -- the backward update for callers that cannot allocate device
memory (a runtime that plans every allocation at start-up, an allocator the calling layer
cannot reach, code that must not call cudaMalloc) -- checked through the C-ABI against the
workspace entry point tbe_backward_update on two calls in a row.

This file is collected last so that a run stopping at the first failure has already run
every other test; it needs nothing from them and passes on its own in a fresh process."""
import ctypes
import dataclasses

import numpy as np
import pytest
import torch

from bwd_tbe_fwd_gb300 import TBEOptions
from bwd_tbe_fwd_gb300 import tbe as tbe_mod
from synth import get_config
from tbe_harness import Case, weights_f64

pytestmark = pytest.mark.gpu


def _both_entry_points(case, options, calls=2):
    cfg = case.cfg
    w_a, w_b = case.w0.cuda(), case.w0.cuda()
    s_a = torch.zeros(cfg.total_rows, dtype=torch.float32, device="cuda")
    s_b = torch.zeros_like(s_a)
    grad = case.grad.cuda()
    results = []
    for _ in range(calls):
        case.tbe.backward_update(w_a, s_a, case.idx_d, case.off_d, grad, psw=case.psw_d, optimizer="adagrad",
                                 lr=cfg.lr, eps=cfg.eps, options=options)
        tbe_mod.tbe_backward_update_noalloc(case.tbe, w_b, s_b, case.idx_d, case.off_d, grad, psw=case.psw_d,
                                            optimizer="adagrad", lr=cfg.lr, eps=cfg.eps, options=options)
        torch.cuda.synchronize()
        results.append((weights_f64(w_a), weights_f64(w_b), s_a.cpu().numpy().copy(), s_b.cpu().numpy().copy()))
    return results


def test_noalloc_matches_workspace_entry_point_fp32_with_long_runs():
    # fp32 tables (rtol 1e-5) with skewed ids, so long runs take the atomic split-256 path
    cfg = dataclasses.replace(get_config("c3").shrink(B=2048, T=4, E_div=4000), wdtype="f32", w_scale=0.1,
                              name="noalloc_f32")
    case = Case(cfg)
    assert case.tbe.ws_backward.numel() <= tbe_mod.TBE_STATIC_SCRATCH_BYTES
    opts = TBEOptions()
    for w_a, w_b, s_a, s_b in _both_entry_points(case, opts):
        assert not np.array_equal(w_a, weights_f64(case.w0))
        rows = w_a.reshape(-1, 128)
        floor = np.abs(rows).max(axis=1, keepdims=True) / 64.0
        bound = 1e-5 * np.maximum(np.abs(rows), floor)
        assert np.all(np.abs(w_b.reshape(-1, 128) - rows) <= bound)
        assert np.all(np.abs(s_b - s_a) <= 1e-5 * np.maximum(s_a, 1e-30))
    m = case.tbe.metadata()
    assert m["num_long"] > 0


def test_noalloc_is_bitwise_equal_when_every_run_is_short():
    # weighted bf16 tables with every run on the atomic-free short path: both entry points
    # compute in the same order, so the results agree bit for bit on both calls
    cfg = get_config("c5").shrink(B=256, E_div=100)
    opts = TBEOptions(long_threshold=1 << 30)
    case = Case(cfg, options=opts)
    assert case.tbe.ws_backward.numel() <= tbe_mod.TBE_STATIC_SCRATCH_BYTES
    for w_a, w_b, s_a, s_b in _both_entry_points(case, opts):
        assert np.array_equal(w_a, w_b)
        assert np.array_equal(s_a, s_b)


def test_noalloc_rejects_problems_beyond_the_scratch_size():
    lib = tbe_mod.load()
    D = (ctypes.c_int32 * 1)(128)
    E = (ctypes.c_int64 * 1)(1_000_000)
    prob = tbe_mod.Problem(1, 100_000, 50_000_000, D, E, tbe_mod.TBE_F16, tbe_mod.TBE_I64, 0, None)
    fn = lib.tbe_backward_update_noalloc
    fn.argtypes = [ctypes.POINTER(tbe_mod.Problem), ctypes.c_void_p, ctypes.c_void_p] + [ctypes.c_void_p] * 6 + \
        [ctypes.c_int, ctypes.c_float, ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    lib.tbe_backward_workspace_size.argtypes = [ctypes.POINTER(tbe_mod.Problem), ctypes.c_void_p]
    lib.tbe_backward_workspace_size.restype = ctypes.c_size_t
    assert lib.tbe_backward_workspace_size(ctypes.byref(prob), None) > tbe_mod.TBE_STATIC_SCRATCH_BYTES
    # every data pointer NULL: the size check rejects the call first; were it ever to pass, the
    # workspace entry point's argument checks would reject the NULL buffers before any launch
    tables = tbe_mod.Tables(None, None, None)
    st = fn(ctypes.byref(prob), None, ctypes.byref(tables), None, None, None, None, None, None,
            tbe_mod.TBE_OPT_ROWWISE_ADAGRAD, 0.01, 1e-8, None, None)
    assert st == tbe_mod.TBE_ERR_WORKSPACE
    # an invalid problem gets the status the workspace entry point gives it
    bad = tbe_mod.Problem(0, 100, 1000, D, E, tbe_mod.TBE_F16, tbe_mod.TBE_I64, 0, None)
    st = fn(ctypes.byref(bad), None, ctypes.byref(tables), None, None, None, None, None, None,
            tbe_mod.TBE_OPT_ROWWISE_ADAGRAD, 0.01, 1e-8, None, None)
    assert st == lib.tbe_backward_update(ctypes.byref(bad), None, ctypes.byref(tables), None, None, None, None,
                                         None, None, tbe_mod.TBE_OPT_ROWWISE_ADAGRAD, ctypes.c_float(0.01),
                                         ctypes.c_float(1e-8), None, 0, None, None) != tbe_mod.TBE_OK
