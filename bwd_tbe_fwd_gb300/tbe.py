"""ctypes binding of the C interface in include/tbe.h.

Argument marshalling only: every step of the forward and backward runs in the CUDA library
``libtbe_gb300.so``; torch supplies device memory (weights, workspaces) and the current
stream.  If the library is missing or does not load, every entry point raises -- there is no
other implementation to fall back on.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

c_i32, c_i64, c_u8, c_f32, vp = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint8, ctypes.c_float, ctypes.c_void_p

TBE_OK, TBE_ERR_INVALID_ARG, TBE_ERR_UNSUPPORTED, TBE_ERR_WORKSPACE, TBE_ERR_CUDA, TBE_ERR_RANGE = range(6)
TBE_F32, TBE_F16, TBE_BF16 = 0, 1, 2
TBE_I32, TBE_I64 = 0, 1
TBE_POOL_SUM, TBE_POOL_MEAN = 0, 1
TBE_OPT_SGD, TBE_OPT_ROWWISE_ADAGRAD = 0, 1
TBE_LONG_AUTO, TBE_LONG_TWO_KERNEL, TBE_LONG_FUSED = 0, 1, 2
TBE_SCHED_GRID, TBE_SCHED_PERSISTENT, TBE_SCHED_CLC = 0, 1, 2
TBE_MERGE_ATOMIC, TBE_MERGE_BULK = 0, 1
TBE_GATHER_REGISTER, TBE_GATHER_TMA = 0, 1
TBE_CLASSIFY_ATOMIC, TBE_CLASSIFY_ORDERED = 0, 1
TBE_FWD_NUM_EVENTS = 3
TBE_BWD_NUM_EVENTS = 9
FWD_STAGES = ("gather", "histogram")
BWD_STAGES = ("expand", "sort", "rle", "classify", "short", "long", "apply", "bwd_histogram")
TBE_NUM_STATS = 8
STAT_NAMES = ("bad_indices", "bad_offsets", "unrepaired", "wait_timeout", "check_failed")
TBE_CNT_N, TBE_CNT_RUNS, TBE_CNT_LONG, TBE_CNT_CHUNKS, TBE_CNT_SHORT0 = 0, 1, 2, 3, 4
TBE_NUM_BUCKETS = 11
TBE_NUM_COUNTERS = 32

EXPORTED = (
    "tbe_default_options", "tbe_table_layout", "tbe_bounds_workspace_size", "tbe_bounds_check",
    "tbe_forward_workspace_size", "tbe_forward", "tbe_backward_workspace_size",
    "tbe_backward_update", "tbe_backward_metadata", "tbe_status_string", "tbe_version",
    "tbe_last_cuda_error", "tbe_backward_update_noalloc", "tbe_backward_prepare", "tbe_psw_gradient",
    "tbe_bounds_check_offsets", "tbe_selftest_wait_timeout",
)
TBE_STATIC_SCRATCH_BYTES = 64 * 1024 * 1024


class Problem(ctypes.Structure):
    _fields_ = [("T", c_i32), ("B", c_i64), ("num_indices", c_i64), ("D", ctypes.POINTER(c_i32)),
                ("E", ctypes.POINTER(c_i64)), ("wdtype", ctypes.c_int), ("itype", ctypes.c_int),
                ("weighted", c_i32), ("long_bags", ctypes.POINTER(c_u8)), ("pooling", c_i32)]


class Tables(ctypes.Structure):
    _fields_ = [("weight_offsets", vp), ("D_offsets", vp), ("row_offsets", vp)]


class Options(ctypes.Structure):
    _fields_ = [("long_threshold", c_i32), ("chunk", c_i32), ("long_mode", c_i32), ("scheduler", c_i32),
                ("histogram", c_i32), ("fused_bounds", c_i32), ("events", ctypes.POINTER(vp)),
                ("num_events", c_i32), ("launch_counter", ctypes.POINTER(c_i64)), ("classify_mode", c_i32),
                ("prepared", c_i32), ("merge", c_i32), ("gather", c_i32), ("nvtx", c_i32),
                ("forward_ws", vp)]


class RunMetadata(ctypes.Structure):
    _fields_ = [(n, vp) for n in ("counters", "sorted_keys", "sorted_bags", "sorted_psw", "unique_keys",
                                  "run_offsets", "run_lengths", "long_runs")]


class TBEError(RuntimeError):
    pass


_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return _build.LIB_PATH


def load(path: str | None = None):
    """Loads the CUDA library (raises if it is missing: build it with bwd_tbe_fwd_gb300.build)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or _build.LIB_PATH
        if not os.path.exists(p):
            raise TBEError(f"TBE CUDA library not found at {p}; run bwd_tbe_fwd_gb300.build.build()")
        lib = ctypes.CDLL(p)
        P, T, O, M = (ctypes.POINTER(x) for x in (Problem, Tables, Options, RunMetadata))
        lib.tbe_default_options.argtypes = [O]
        lib.tbe_default_options.restype = None
        lib.tbe_table_layout.argtypes = [P, vp, vp, vp]
        lib.tbe_bounds_workspace_size.argtypes = [P]
        lib.tbe_bounds_workspace_size.restype = ctypes.c_size_t
        lib.tbe_bounds_check.argtypes = [P, T, vp, vp, vp, ctypes.c_size_t, vp, vp]
        lib.tbe_bounds_check_offsets.argtypes = [P, T, vp, vp, ctypes.c_size_t, vp, vp]
        lib.tbe_forward_workspace_size.argtypes = [P, O]
        lib.tbe_forward_workspace_size.restype = ctypes.c_size_t
        lib.tbe_forward.argtypes = [P, O, T, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, vp, vp]
        lib.tbe_backward_workspace_size.argtypes = [P, O]
        lib.tbe_backward_workspace_size.restype = ctypes.c_size_t
        lib.tbe_backward_update.argtypes = [P, O, T, vp, vp, vp, vp, vp, vp, ctypes.c_int, c_f32, c_f32,
                                            vp, ctypes.c_size_t, vp, vp]
        lib.tbe_backward_prepare.argtypes = [P, O, T, vp, vp, vp, vp, ctypes.c_size_t, vp, vp]
        lib.tbe_psw_gradient.argtypes = [P, O, T, vp, vp, vp, vp, vp, vp]
        lib.tbe_backward_metadata.argtypes = [P, O, vp, ctypes.c_size_t, M]
        lib.tbe_status_string.argtypes = [ctypes.c_int]
        lib.tbe_status_string.restype = ctypes.c_char_p
        lib.tbe_version.restype = ctypes.c_int
        lib.tbe_last_cuda_error.restype = ctypes.c_int
        for name in ("tbe_table_layout", "tbe_bounds_check", "tbe_bounds_check_offsets", "tbe_forward",
                     "tbe_backward_update",
                     "tbe_backward_prepare", "tbe_psw_gradient", "tbe_backward_metadata"):
            getattr(lib, name).restype = ctypes.c_int
        if path is None:
            _lib = lib
        return lib


def _check(lib, status: int, what: str):
    if status != TBE_OK:
        msg = lib.tbe_status_string(status).decode()
        if status == TBE_ERR_CUDA:
            msg += f" (cudaError {lib.tbe_last_cuda_error()})"
        raise TBEError(f"{what} failed: {msg}")


def _ptr(t: torch.Tensor | None):
    return None if t is None else vp(t.data_ptr())


def _stream(stream, device) -> vp:
    """The cudaStream_t of `stream`, or of the current stream of `device` when None."""
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return vp(s.cuda_stream)


_WDTYPE = {torch.float32: TBE_F32, torch.float16: TBE_F16, torch.bfloat16: TBE_BF16}
_ITYPE = {torch.int32: TBE_I32, torch.int64: TBE_I64}


class TBEOptions:
    """Python view of tbe_options (defaults from the library)."""

    def __init__(self, **kw):
        self.c = Options()
        load().tbe_default_options(ctypes.byref(self.c))
        self._events = None
        for k, v in kw.items():
            if not hasattr(self.c, k):
                raise TypeError(f"unknown option {k}")
            setattr(self.c, k, v)

    def count_launches(self, counter: "ctypes.c_int64 | None"):
        """Have the library add its kernel launches to a host int64 (ctypes.c_int64)."""
        self._counter = counter
        self.c.launch_counter = None if counter is None else ctypes.pointer(counter)
        return self

    def with_events(self, events: list | None):
        """Record CUDA events (torch.cuda.Event) at stage ends; None clears."""
        if events is None:
            self.c.events = None
            self.c.num_events = 0
            self._events = None
        else:
            for e in events:  # torch creates the CUDA event on its first record
                if e is not None and e.cuda_event == 0:
                    e.record()
            arr = (vp * len(events))(*[vp(e.cuda_event) if e is not None else None for e in events])
            self._events = (arr, events)
            self.c.events = ctypes.cast(arr, ctypes.POINTER(vp))
            self.c.num_events = len(events)
        return self


class TableBatchedEmbedding:
    """One problem shape (tables, batch size, index capacity) with its device layout arrays and
    caller-owned workspaces, and the three operations of the library.  Every call runs with the
    problem's device current (the library launches on the current device) and on the stream
    passed, else on that device's current stream."""

    def __init__(self, D, E, B: int, num_indices: int, weight_dtype: torch.dtype,
                 index_dtype: torch.dtype = torch.int64, weighted: bool = False, long_bags=None,
                 device="cuda", options: TBEOptions | None = None, pooling: str = "sum"):
        self.lib = load()
        dev = torch.device(device)
        if dev.type == "cuda" and dev.index is None:
            dev = torch.device("cuda", torch.cuda.current_device())
        self.device = dev
        self.D = [int(d) for d in D]
        self.E = [int(e) for e in E]
        self.T = len(self.D)
        self.B = int(B)
        self.num_indices = int(num_indices)
        self.weight_dtype = weight_dtype
        self.index_dtype = index_dtype
        self.weighted = bool(weighted)
        self._D = (c_i32 * self.T)(*self.D)
        self._E = (c_i64 * self.T)(*self.E)
        self._long = (c_u8 * self.T)(*([1 if x else 0 for x in long_bags] if long_bags is not None else [0] * self.T))
        self.pooling = pooling
        self.prob = Problem(self.T, self.B, self.num_indices, self._D, self._E, _WDTYPE[weight_dtype],
                            _ITYPE[index_dtype], 1 if self.weighted else 0, self._long,
                            {"sum": TBE_POOL_SUM, "mean": TBE_POOL_MEAN}[pooling])
        self.options = options or TBEOptions()
        woff = (c_i64 * (self.T + 1))()
        doff = (c_i32 * (self.T + 1))()
        roff = (c_i64 * (self.T + 1))()
        _check(self.lib, self.lib.tbe_table_layout(ctypes.byref(self.prob), woff, doff, roff), "tbe_table_layout")
        self.weight_offsets = torch.tensor(list(woff), dtype=torch.int64, device=self.device)
        self.D_offsets = torch.tensor(list(doff), dtype=torch.int32, device=self.device)
        self.row_offsets = torch.tensor(list(roff), dtype=torch.int64, device=self.device)
        self.num_weights = int(woff[self.T])
        self.total_rows = int(roff[self.T])
        self.total_D = int(doff[self.T])
        self.tables = Tables(self.weight_offsets.data_ptr(), self.D_offsets.data_ptr(), self.row_offsets.data_ptr())
        with torch.cuda.device(self.device):
            nb = self.lib.tbe_bounds_workspace_size(ctypes.byref(self.prob))
            nf = self.lib.tbe_forward_workspace_size(ctypes.byref(self.prob), ctypes.byref(self.options.c))
            nw = self.lib.tbe_backward_workspace_size(ctypes.byref(self.prob), ctypes.byref(self.options.c))
        if nw == 0:
            raise TBEError("tbe_backward_workspace_size rejected the problem")
        self.ws_bounds = torch.empty(max(nb, 256), dtype=torch.uint8, device=self.device)
        self.ws_forward = torch.empty(max(nf, 256), dtype=torch.uint8, device=self.device)
        self.ws_backward = torch.empty(nw, dtype=torch.uint8, device=self.device)

    # -- checks -----------------------------------------------------------------------------
    def _idx(self, indices: torch.Tensor, offsets: torch.Tensor):
        if indices.dtype != self.index_dtype or offsets.dtype != self.index_dtype:
            raise TypeError("indices/offsets dtype does not match the problem")
        if indices.numel() != self.num_indices or offsets.numel() != self.T * self.B + 1:
            raise ValueError("indices/offsets sizes do not match the problem")
        for t in (indices, offsets):
            if t.device != self.device or not t.is_contiguous():
                raise ValueError("indices/offsets must be contiguous on the problem's device")

    def _dev(self, t: torch.Tensor | None, name: str, dtype=None, numel=None):
        if t is None:
            return
        if t.device != self.device or not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous on {self.device}")
        if dtype is not None and t.dtype != dtype:
            raise TypeError(f"{name} must be {dtype}")
        if numel is not None and t.numel() != numel:
            raise ValueError(f"{name} must have {numel} elements")

    # -- operations --------------------------------------------------------------------------
    def bounds_check(self, indices, offsets, stats=None, stream=None, offsets_only: bool = False):
        """Repairs offsets and ids in place; offsets_only leaves the ids to a forward with
        fused_bounds=1."""
        self._idx(indices, offsets)
        self._dev(stats, "stats", torch.int64, TBE_NUM_STATS)
        with torch.cuda.device(self.device):
            if offsets_only:
                st = self.lib.tbe_bounds_check_offsets(ctypes.byref(self.prob), ctypes.byref(self.tables),
                                                       _ptr(offsets), _ptr(self.ws_bounds), self.ws_bounds.numel(),
                                                       _ptr(stats), _stream(stream, self.device))
                _check(self.lib, st, "tbe_bounds_check_offsets")
                return
            st = self.lib.tbe_bounds_check(ctypes.byref(self.prob), ctypes.byref(self.tables), _ptr(indices),
                                           _ptr(offsets), _ptr(self.ws_bounds), self.ws_bounds.numel(),
                                           _ptr(stats), _stream(stream, self.device))
        _check(self.lib, st, "tbe_bounds_check")

    def forward(self, weights, indices, offsets, psw=None, out=None, stats=None, stream=None,
                options: TBEOptions | None = None):
        self._idx(indices, offsets)
        self._dev(weights, "weights", self.weight_dtype, self.num_weights)
        self._dev(psw, "psw", torch.float32, self.num_indices)
        self._dev(stats, "stats", torch.int64, TBE_NUM_STATS)
        if out is None:
            out = torch.empty(self.B, self.total_D, dtype=torch.float32, device=self.device)
        self._dev(out, "out", torch.float32, self.B * self.total_D)
        o = (options or self.options).c
        with torch.cuda.device(self.device):
            st = self.lib.tbe_forward(ctypes.byref(self.prob), ctypes.byref(o), ctypes.byref(self.tables),
                                      _ptr(weights), _ptr(indices), _ptr(offsets), _ptr(psw), _ptr(out),
                                      _ptr(self.ws_forward), self.ws_forward.numel(), _ptr(stats),
                                      _stream(stream, self.device))
        _check(self.lib, st, "tbe_forward")
        return out

    def psw_gradient(self, weights, indices, offsets, grad_out, grad_psw=None, stream=None,
                     options: TBEOptions | None = None):
        """Gradient with respect to the per-sample weights (weighted problems); call it before
        backward_update changes the weights.  Returns grad_psw [num_indices] fp32."""
        self._idx(indices, offsets)
        self._dev(weights, "weights", self.weight_dtype, self.num_weights)
        self._dev(grad_out, "grad_out", torch.float32, self.B * self.total_D)
        if grad_psw is None:
            grad_psw = torch.zeros(self.num_indices, dtype=torch.float32, device=self.device)
        self._dev(grad_psw, "grad_psw", torch.float32, self.num_indices)
        o = (options or self.options).c
        with torch.cuda.device(self.device):
            st = self.lib.tbe_psw_gradient(ctypes.byref(self.prob), ctypes.byref(o), ctypes.byref(self.tables),
                                           _ptr(weights), _ptr(indices), _ptr(offsets), _ptr(grad_out),
                                           _ptr(grad_psw), _stream(stream, self.device))
        _check(self.lib, st, "tbe_psw_gradient")
        return grad_psw

    def backward_prepare(self, indices, offsets, psw=None, stats=None, stream=None,
                         options: TBEOptions | None = None):
        """The transpose half of the backward (linearize, sort, RLE, classify) into the backward
        workspace; a following backward_update with prepared=True only applies the updates."""
        self._idx(indices, offsets)
        self._dev(psw, "psw", torch.float32, self.num_indices)
        self._dev(stats, "stats", torch.int64, TBE_NUM_STATS)
        o = (options or self.options).c
        if o.long_threshold != self.options.c.long_threshold or o.chunk != self.options.c.chunk:
            raise ValueError("threshold/chunk differ from the options the workspace was sized for")
        with torch.cuda.device(self.device):
            st = self.lib.tbe_backward_prepare(
                ctypes.byref(self.prob), ctypes.byref(o), ctypes.byref(self.tables), _ptr(indices), _ptr(offsets),
                _ptr(psw), _ptr(self.ws_backward), self.ws_backward.numel(), _ptr(stats),
                _stream(stream, self.device))
        _check(self.lib, st, "tbe_backward_prepare")

    def backward_update(self, weights, state, indices, offsets, grad_out, psw=None, optimizer="adagrad",
                        lr=0.01, eps=1e-8, stats=None, stream=None, options: TBEOptions | None = None,
                        prepared: bool = False, reuse_forward: bool = False):
        """reuse_forward: the last forward() of this object ran on the same batch (indices and
        offsets unchanged since): its counts x table tables' per-bag counts, saved in the forward
        workspace, replace reading their ids again (tbe_options.forward_ws)."""
        self._idx(indices, offsets)
        self._dev(weights, "weights", self.weight_dtype, self.num_weights)
        self._dev(state, "state", torch.float32, self.total_rows)
        self._dev(grad_out, "grad_out", torch.float32, self.B * self.total_D)
        self._dev(psw, "psw", torch.float32, self.num_indices)
        self._dev(stats, "stats", torch.int64, TBE_NUM_STATS)
        opt = {"sgd": TBE_OPT_SGD, "adagrad": TBE_OPT_ROWWISE_ADAGRAD}[optimizer]
        o = (options or self.options).c
        if o.long_threshold != self.options.c.long_threshold or o.chunk != self.options.c.chunk:
            raise ValueError("threshold/chunk differ from the options the workspace was sized for")
        if bool(o.prepared) != prepared or reuse_forward:
            o = Options.from_buffer_copy(o)
            o.prepared = 1 if prepared else 0
            if reuse_forward:
                o.forward_ws = self.ws_forward.data_ptr()
        with torch.cuda.device(self.device):
            st = self.lib.tbe_backward_update(
                ctypes.byref(self.prob), ctypes.byref(o), ctypes.byref(self.tables), _ptr(weights), _ptr(state),
                _ptr(indices), _ptr(offsets), _ptr(psw), _ptr(grad_out), opt, c_f32(lr), c_f32(eps),
                _ptr(self.ws_backward), self.ws_backward.numel(), _ptr(stats), _stream(stream, self.device))
        _check(self.lib, st, "tbe_backward_update")

    def metadata(self) -> dict:
        """Run metadata of the last backward (synchronizes to read the device counts)."""
        m = RunMetadata()
        st = self.lib.tbe_backward_metadata(ctypes.byref(self.prob), ctypes.byref(self.options.c),
                                            _ptr(self.ws_backward), self.ws_backward.numel(), ctypes.byref(m))
        _check(self.lib, st, "tbe_backward_metadata")
        base = self.ws_backward.data_ptr()

        def view(ptr, n, dtype):
            off = ptr - base
            esz = torch.tensor([], dtype=dtype).element_size()
            return self.ws_backward[off:off + n * esz].view(dtype)

        counters_device = view(m.counters, TBE_NUM_COUNTERS, torch.int32)
        counters = counters_device.clone().cpu().numpy().view("uint32")
        N, U, nlong = int(counters[TBE_CNT_N]), int(counters[TBE_CNT_RUNS]), int(counters[TBE_CNT_LONG])
        out = dict(
            counters=counters, counters_device=counters_device, N=N, U=U, num_long=nlong, num_chunks=int(counters[TBE_CNT_CHUNKS]),
            short_per_bucket=counters[TBE_CNT_SHORT0:TBE_CNT_SHORT0 + TBE_NUM_BUCKETS].copy(),
            sorted_keys=view(m.sorted_keys, N, torch.int32), sorted_bags=view(m.sorted_bags, N, torch.int32),
            unique_keys=view(m.unique_keys, U, torch.int32), run_offsets=view(m.run_offsets, U + 1, torch.int32),
            run_lengths=view(m.run_lengths, U, torch.int32), long_runs=view(m.long_runs, nlong, torch.int32))
        if m.sorted_psw:
            out["sorted_psw"] = view(m.sorted_psw, N, torch.float32)
        return out


# Module-level names mirroring the C interface.
def tbe_bounds_check(tbe: TableBatchedEmbedding, *a, **k):
    return tbe.bounds_check(*a, **k)


def tbe_forward(tbe: TableBatchedEmbedding, *a, **k):
    return tbe.forward(*a, **k)


def tbe_backward_update(tbe: TableBatchedEmbedding, *a, **k):
    return tbe.backward_update(*a, **k)


def tbe_backward_metadata(tbe: TableBatchedEmbedding):
    return tbe.metadata()


def tbe_backward_update_noalloc(tbe: TableBatchedEmbedding, weights, state, indices, offsets, grad_out,
                                psw=None, optimizer="adagrad", lr=0.01, eps=1e-8, stats=None, stream=None,
                                options: TBEOptions | None = None):
    """The backward update for callers that cannot allocate device memory: same arguments as
    TableBatchedEmbedding.backward_update, but the library uses its built-in scratch array
    (TBE_STATIC_SCRATCH_BYTES) instead of a workspace.  Problems whose workspace would exceed
    that size raise; calls on one device share the array and must not overlap on the GPU."""
    lib = tbe.lib
    fn = lib.tbe_backward_update_noalloc
    fn.argtypes = [ctypes.POINTER(Problem), ctypes.POINTER(Options), ctypes.POINTER(Tables), vp, vp, vp, vp,
                   vp, vp, ctypes.c_int, c_f32, c_f32, vp, vp]
    fn.restype = ctypes.c_int
    tbe._idx(indices, offsets)
    tbe._dev(weights, "weights", tbe.weight_dtype, tbe.num_weights)
    tbe._dev(state, "state", torch.float32, tbe.total_rows)
    tbe._dev(grad_out, "grad_out", torch.float32, tbe.B * tbe.total_D)
    tbe._dev(psw, "psw", torch.float32, tbe.num_indices)
    tbe._dev(stats, "stats", torch.int64, TBE_NUM_STATS)
    opt = {"sgd": TBE_OPT_SGD, "adagrad": TBE_OPT_ROWWISE_ADAGRAD}[optimizer]
    o = (options or tbe.options).c
    with torch.cuda.device(tbe.device):
        st = fn(ctypes.byref(tbe.prob), ctypes.byref(o), ctypes.byref(tbe.tables), _ptr(weights), _ptr(state),
                _ptr(indices), _ptr(offsets), _ptr(psw), _ptr(grad_out), opt, c_f32(lr), c_f32(eps), _ptr(stats),
                _stream(stream, tbe.device))
    _check(lib, st, "tbe_backward_update_noalloc")


def selftest_wait_timeout(stats: torch.Tensor, polls: int = 8, stream=None):
    """Diagnostic: one CTA waits, through the library's bounded mbarrier wait, for a phase that
    never completes; it gives up after `polls` polls and adds 1 to stats[TBE_STAT_WAIT_TIMEOUT]
    (stats: device int64[TBE_NUM_STATS]).  Asynchronous on `stream` (default: the current one)."""
    lib = load()
    fn = lib.tbe_selftest_wait_timeout
    fn.argtypes = [ctypes.c_uint32, vp, vp]
    fn.restype = ctypes.c_int
    if not (stats.is_cuda and stats.dtype == torch.int64 and stats.numel() >= TBE_NUM_STATS):
        raise TBEError(f"stats must be a CUDA int64 tensor of at least {TBE_NUM_STATS} elements")
    with torch.cuda.device(stats.device):
        st = fn(polls, _ptr(stats), _stream(stream, stats.device))
    _check(lib, st, "tbe_selftest_wait_timeout")
