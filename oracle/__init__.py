"""CPU oracle for the table-batched embedding (TBE) forward and backward pass.

TEST INFRASTRUCTURE ONLY.  This package wraps ``tbe_oracle.cpp`` -- a plain, slow,
single-threaded C++ implementation with fp64 accumulation and a ``std::map`` grouping -- so
that the tests, the smoke check and the CPU-baseline leg of ``bench.py`` can compare the
CUDA library against it.  Nothing on the product path imports this package, and it imports
nothing from the product (``bwd_tbe_fwd_gb300``).

Array conventions (numpy):
  * weights: the packed tables (table t after all rows of tables < t), as ``float32``,
    ``float16``, or ``uint16`` holding bfloat16 bit patterns (pass ``wdtype="bf16"``).
  * indices / offsets: ``int32`` or ``int64`` (both the same), offsets table-major of
    length T*B+1.
  * psw: ``float32`` per index or None; grad_out / pooled output: ``float32`` [B, sum(D)].

Parity of every function here is pinned in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tbe_oracle.cpp")
_HDR = os.path.join(_HERE, "tbe_oracle.h")
_LIB = os.path.join(_HERE, "liboracle_tbe.so")
_lock = threading.Lock()
_lib = None

WDTYPES = {"f32": 0, "f16": 1, "bf16": 2}
NUM_BUCKETS = 11

# -ffp-contract=off: the oracle is the plain reading of the formulas, one rounding per
# operation on every host (GCC would otherwise fuse multiply-adds on aarch64).
CXXFLAGS = ["-O2", "-std=c++17", "-fPIC", "-shared", "-ffp-contract=off", "-Wall", "-Wextra"]


def build(force: bool = False, out: str | None = None, extra_flags: list[str] | None = None,
          src: str | None = None) -> str:
    """Compile the oracle into a shared library (g++), unless it is up to date."""
    out = out or _LIB
    src = src or _SRC
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= max(os.path.getmtime(src), os.path.getmtime(_HDR))):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["g++", *CXXFLAGS, *(extra_flags or []), "-I", _HERE, src, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _bind(lib):
    c_i32, c_i64, c_f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    vp = ctypes.c_void_p
    lib.oracle_version.restype = ctypes.c_int
    lib.oracle_bounds_repair.argtypes = [c_i32, c_i64, c_i64, vp, c_i32, vp, vp, vp, vp]
    lib.oracle_bounds_repair.restype = ctypes.c_int
    lib.oracle_forward.argtypes = [c_i32, c_i64, vp, vp, c_i32, vp, c_i32, vp, vp, vp, c_i32, vp, vp, vp]
    lib.oracle_forward.restype = ctypes.c_int
    lib.oracle_backward.argtypes = [c_i32, c_i64, vp, vp, c_i32, vp, vp, c_i32, vp, vp, vp, vp,
                                    c_i32, c_i32, c_f32, c_f32, vp]
    lib.oracle_psw_gradient.argtypes = [c_i32, c_i64, vp, vp, c_i32, vp, c_i32, vp, vp, vp, c_i32, vp]
    lib.oracle_psw_gradient.restype = ctypes.c_int
    lib.oracle_backward.restype = vp
    for name in ("oracle_result_num_lookups", "oracle_result_num_runs", "oracle_result_num_elems"):
        getattr(lib, name).argtypes = [vp]
        getattr(lib, name).restype = c_i64
    lib.oracle_result_copy.argtypes = [vp] * 12
    lib.oracle_result_copy.restype = None
    lib.oracle_result_free.argtypes = [vp]
    lib.oracle_result_free.restype = None
    lib.oracle_classify.argtypes = [c_i32, vp, vp, c_i64, vp, vp, c_i64, c_i64, vp, vp, vp, vp]
    lib.oracle_classify.restype = ctypes.c_int
    lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_half_to_double.restype = ctypes.c_double
    lib.oracle_double_to_half.argtypes = [ctypes.c_double]
    lib.oracle_double_to_half.restype = ctypes.c_uint16
    lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_double.restype = ctypes.c_double
    lib.oracle_double_to_bf16.argtypes = [ctypes.c_double]
    lib.oracle_double_to_bf16.restype = ctypes.c_uint16
    return lib


def load(path: str | None = None):
    """Load (building first if needed) the oracle library; ``path`` loads another build."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _ptr(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _itype(indices, offsets):
    if indices.dtype != offsets.dtype or indices.dtype not in (np.int32, np.int64):
        raise TypeError("indices and offsets must share one dtype, int32 or int64")
    return 0 if indices.dtype == np.int32 else 1


_POOL = {"sum": 0, "mean": 1}


def _wdtype(weights, wdtype):
    if wdtype is None:
        wdtype = {np.dtype(np.float32): "f32", np.dtype(np.float16): "f16"}.get(weights.dtype)
    if wdtype not in WDTYPES:
        raise TypeError("weights must be float32, float16, or uint16 bf16 bits with wdtype='bf16'")
    want = {"f32": np.float32, "f16": np.float16, "bf16": np.uint16}[wdtype]
    if weights.dtype != want:
        raise TypeError(f"weights dtype {weights.dtype} does not match wdtype {wdtype}")
    return WDTYPES[wdtype]


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


class Tables:
    """Per-table sizes: D[t] (row width) and E[t] (rows)."""

    def __init__(self, D, E):
        self.D = _c(D, np.int32)
        self.E = _c(E, np.int64)
        if self.D.shape != self.E.shape or self.D.ndim != 1:
            raise ValueError("D and E must be 1-D of equal length")
        self.T = int(self.D.shape[0])


class Oracle:
    """The oracle functions bound to one build of the library (the default build, or a
    modified copy compiled by a test)."""

    def __init__(self, lib):
        self.lib = lib

    def bounds_repair(self, tables: Tables, B: int, indices: np.ndarray, offsets: np.ndarray,
                      num_indices: int | None = None):
        """Repairs indices/offsets in place; returns (repaired per table [T], repaired offsets)."""
        lib = self.lib
        it = _itype(indices, offsets)
        assert indices.flags.c_contiguous and offsets.flags.c_contiguous
        per_table = np.zeros(tables.T, dtype=np.int64)
        n_off = np.zeros(1, dtype=np.int64)
        n = int(indices.shape[0]) if num_indices is None else int(num_indices)
        rc = lib.oracle_bounds_repair(tables.T, B, n, _ptr(tables.E), it, _ptr(indices), _ptr(offsets),
                                      _ptr(per_table), _ptr(n_off))
        if rc != 0:
            raise RuntimeError(f"oracle_bounds_repair failed: {rc}")
        return per_table, int(n_off[0])

    def forward(self, tables: Tables, B: int, weights: np.ndarray, indices: np.ndarray, offsets: np.ndarray,
                psw: np.ndarray | None = None, wdtype: str | None = None, pooling: str = "sum"):
        """Returns (out fp32, out_exact fp64, out_absterms fp64), each [B, sum(D)]."""
        lib = self.lib
        wd = _wdtype(weights, wdtype)
        it = _itype(indices, offsets)
        width = int(tables.D.sum())
        out = np.empty((B, width), dtype=np.float32)
        exact = np.empty((B, width), dtype=np.float64)
        absterms = np.empty((B, width), dtype=np.float64)
        psw_c = None if psw is None else _c(psw, np.float32)
        rc = lib.oracle_forward(tables.T, B, _ptr(tables.D), _ptr(tables.E), wd, _ptr(_c(weights, weights.dtype)),
                                it, _ptr(_c(indices, indices.dtype)), _ptr(_c(offsets, offsets.dtype)),
                                _ptr(psw_c), _POOL[pooling], _ptr(out), _ptr(exact), _ptr(absterms))
        if rc != 0:
            raise RuntimeError(f"oracle_forward failed: {rc}")
        return out, exact, absterms

    def psw_gradient(self, tables: Tables, B: int, weights: np.ndarray, indices: np.ndarray, offsets: np.ndarray,
                     grad_out: np.ndarray, wdtype: str | None = None, pooling: str = "sum") -> np.ndarray:
        """fp64 gradient with respect to the per-sample weights, one value per index position
        (positions outside every bag stay NaN)."""
        lib = self.lib
        wd = _wdtype(weights, wdtype)
        it = _itype(indices, offsets)
        g = np.full(len(indices), np.nan, dtype=np.float64)
        rc = lib.oracle_psw_gradient(tables.T, B, _ptr(tables.D), _ptr(tables.E), wd, _ptr(_c(weights, weights.dtype)),
                                     it, _ptr(_c(indices, indices.dtype)), _ptr(_c(offsets, offsets.dtype)),
                                     _ptr(_c(grad_out, np.float32)), _POOL[pooling], _ptr(g))
        if rc != 0:
            raise RuntimeError(f"oracle_psw_gradient failed: {rc}")
        return g

    def backward(self, tables: Tables, B: int, weights: np.ndarray, state: np.ndarray | None,
                 indices: np.ndarray, offsets: np.ndarray, grad_out: np.ndarray,
                 psw: np.ndarray | None = None, optimizer: str = "adagrad", lr: float = 0.01,
                 eps: float = 1e-8, wdtype: str | None = None, pooling: str = "sum") -> dict:
        """Updates weights (and state, for Adagrad) in place; returns the run metadata and
        the exact per-run values as a dict of numpy arrays."""
        lib = self.lib
        wd = _wdtype(weights, wdtype)
        it = _itype(indices, offsets)
        opt = {"sgd": 0, "adagrad": 1}[optimizer]
        assert weights.flags.c_contiguous
        if state is not None:
            assert state.dtype == np.float32 and state.flags.c_contiguous
        grad_c = _c(grad_out, np.float32)
        psw_c = None if psw is None else _c(psw, np.float32)
        status = ctypes.c_int32(0)
        h = lib.oracle_backward(tables.T, B, _ptr(tables.D), _ptr(tables.E), wd, _ptr(weights),
                                _ptr(state), it, _ptr(_c(indices, indices.dtype)),
                                _ptr(_c(offsets, offsets.dtype)), _ptr(psw_c), _ptr(grad_c), _POOL[pooling], opt,
                                ctypes.c_float(lr), ctypes.c_float(eps), ctypes.byref(status))
        if not h:
            raise RuntimeError(f"oracle_backward failed: {status.value}")
        try:
            N = lib.oracle_result_num_lookups(h)
            U = lib.oracle_result_num_runs(h)
            M = lib.oracle_result_num_elems(h)
            r = dict(
                sorted_keys=np.empty(N, np.int64), sorted_bags=np.empty(N, np.int64),
                sorted_psw=np.empty(N, np.float32), unique_keys=np.empty(U, np.int64),
                run_lengths=np.empty(U, np.int64), run_offsets=np.empty(U + 1, np.int64),
                run_elem_offsets=np.empty(U + 1, np.int64), grad_sum=np.empty(M, np.float64),
                w_old=np.empty(M, np.float64), w_exact=np.empty(M, np.float64),
                state_exact=np.empty(U, np.float64))
            lib.oracle_result_copy(h, *(_ptr(r[k]) for k in (
                "sorted_keys", "sorted_bags", "sorted_psw", "unique_keys", "run_lengths", "run_offsets",
                "run_elem_offsets", "grad_sum", "w_old", "w_exact", "state_exact")))
        finally:
            lib.oracle_result_free(h)
        r["num_lookups"] = int(N)
        r["num_runs"] = int(U)
        return r

    def classify(self, tables: Tables, unique_keys: np.ndarray, run_lengths: np.ndarray, threshold: int,
                 chunk: int) -> dict:
        """Run routing: short-run counts per next_pow2(D) bucket, long runs and their chunks."""
        lib = self.lib
        uk = _c(unique_keys, np.int64)
        rl = _c(run_lengths, np.int64)
        U = int(uk.shape[0])
        shorts = np.zeros(NUM_BUCKETS, dtype=np.int64)
        n_long = np.zeros(1, dtype=np.int64)
        n_chunks = np.zeros(1, dtype=np.int64)
        route = np.empty(U, dtype=np.int32)
        rc = lib.oracle_classify(tables.T, _ptr(tables.D), _ptr(tables.E), U, _ptr(uk), _ptr(rl),
                                 int(threshold), int(chunk), _ptr(shorts), _ptr(n_long), _ptr(n_chunks),
                                 _ptr(route))
        if rc != 0:
            raise RuntimeError(f"oracle_classify failed: {rc}")
        return dict(short_per_bucket=shorts, num_short=int(shorts.sum()), num_long=int(n_long[0]),
                    num_chunks=int(n_chunks[0]), route=route)

    def half_to_double(self, bits: int) -> float:
        return self.lib.oracle_half_to_double(bits)

    def double_to_half(self, x: float) -> int:
        return self.lib.oracle_double_to_half(x)

    def bf16_to_double(self, bits: int) -> float:
        return self.lib.oracle_bf16_to_double(bits)

    def double_to_bf16(self, x: float) -> int:
        return self.lib.oracle_double_to_bf16(x)


_default = None


def default() -> Oracle:
    """The oracle bound to the default build (compiled on first use)."""
    global _default
    if _default is None:
        _default = Oracle(load())
    return _default


def bounds_repair(*a, **k):
    return default().bounds_repair(*a, **k)


def forward(*a, **k):
    return default().forward(*a, **k)


def psw_gradient(*a, **k):
    return default().psw_gradient(*a, **k)


def backward(*a, **k):
    return default().backward(*a, **k)


def classify(*a, **k):
    return default().classify(*a, **k)
