"""The C-ABI library on the host: it loads, exports every function include/*.h declares, and
its host-only entry points (layout, options, argument validation) behave as documented.
No call here launches GPU work."""
import ctypes
import os
import re

import pytest

from bwd_tbe_fwd_gb300 import build as tbe_build
from bwd_tbe_fwd_gb300 import tbe

HEADERS = sorted(os.path.join(tbe_build.INCLUDE, f) for f in os.listdir(tbe_build.INCLUDE) if f.endswith(".h"))


@pytest.fixture(scope="module")
def lib():
    tbe_build.build()
    return tbe.load()


def declared_functions():
    names = set()
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"\b(tbe_[a-z_0-9]+)\s*\(", text))
    return sorted(names)


def test_every_declared_function_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 12
    for name in names:
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"
    assert set(names) == set(tbe.EXPORTED)


def _problem(D, E, B=4, n=16, wdtype=tbe.TBE_F16, itype=tbe.TBE_I64, weighted=0):
    Da = (ctypes.c_int32 * len(D))(*D)
    Ea = (ctypes.c_int64 * len(E))(*E)
    p = tbe.Problem(len(D), B, n, Da, Ea, wdtype, itype, weighted, None)
    return p, (Da, Ea)


def test_version_status_and_defaults(lib):
    assert lib.tbe_version() == 1
    assert lib.tbe_status_string(tbe.TBE_ERR_WORKSPACE) == b"workspace too small"
    o = tbe.Options()
    lib.tbe_default_options(ctypes.byref(o))
    assert (o.long_threshold, o.chunk, o.long_mode, o.scheduler, o.histogram, o.fused_bounds) == \
        (256, 256, tbe.TBE_LONG_AUTO, tbe.TBE_SCHED_PERSISTENT, 1, 0)
    assert o.forward_ws is None
    assert (o.classify_mode, o.prepared, o.merge, o.gather, o.nvtx) == \
        (tbe.TBE_CLASSIFY_ORDERED, 0, 0, tbe.TBE_GATHER_REGISTER, 0)


def test_table_layout(lib):
    p, keep = _problem([8, 16, 4], [10, 3, 7])
    w = (ctypes.c_int64 * 4)()
    d = (ctypes.c_int32 * 4)()
    r = (ctypes.c_int64 * 4)()
    assert lib.tbe_table_layout(ctypes.byref(p), w, d, r) == tbe.TBE_OK
    assert list(w) == [0, 80, 128, 156]
    assert list(d) == [0, 8, 24, 28]
    assert list(r) == [0, 10, 13, 20]


@pytest.mark.parametrize("D,E,itype,n,expect", [
    ([6], [10], tbe.TBE_I64, 16, tbe.TBE_ERR_UNSUPPORTED),        # D not a multiple of 4
    ([2048], [10], tbe.TBE_I64, 16, tbe.TBE_ERR_UNSUPPORTED),     # D above 1024
    ([8], [0], tbe.TBE_I64, 16, tbe.TBE_ERR_INVALID_ARG),         # empty table
    ([8], [2 ** 31], tbe.TBE_I32, 16, tbe.TBE_ERR_RANGE),         # int32 ids cannot address the rows
    ([8], [2 ** 31], tbe.TBE_I64, 16, tbe.TBE_ERR_UNSUPPORTED),   # linear keys are 31-bit
    ([8], [10], tbe.TBE_I64, 2 ** 31, tbe.TBE_ERR_UNSUPPORTED),   # lookups beyond 2^31
    ([8], [10], tbe.TBE_I64, 2 ** 31 - 2 ** 16 + 1, tbe.TBE_ERR_UNSUPPORTED),  # within 2^16 of 2^31
    ([8], [10], tbe.TBE_I32, 2 ** 31 - 2 ** 16 + 1, tbe.TBE_ERR_UNSUPPORTED),
    ([8], [10], tbe.TBE_I64, 2 ** 31 - 2 ** 16, tbe.TBE_OK),                   # the largest accepted
    ([8], [10], tbe.TBE_I32, 2 ** 31 - 2 ** 16, tbe.TBE_OK),
])
def test_layout_rejects(lib, D, E, itype, n, expect):
    p, keep = _problem(D, E, itype=itype, n=n)
    assert lib.tbe_table_layout(ctypes.byref(p), None, None, None) == expect


def test_entry_points_validate_before_touching_the_device(lib):
    p, keep = _problem([8], [10])
    t = tbe.Tables(None, None, None)
    # NULL tables / buffers are rejected on the host
    assert lib.tbe_forward(ctypes.byref(p), None, ctypes.byref(t), None, None, None, None, None, None, 0,
                           None, None) == tbe.TBE_ERR_INVALID_ARG
    assert lib.tbe_backward_update(ctypes.byref(p), None, ctypes.byref(t), None, None, None, None, None,
                                   None, tbe.TBE_OPT_SGD, 0.1, 0.0, None, 0, None, None) == tbe.TBE_ERR_INVALID_ARG
    assert lib.tbe_bounds_check(ctypes.byref(p), ctypes.byref(t), None, None, None, 0, None,
                                None) == tbe.TBE_ERR_INVALID_ARG
    # T = 0
    p0, keep0 = _problem([8], [10])
    p0.T = 0
    assert lib.tbe_table_layout(ctypes.byref(p0), None, None, None) == tbe.TBE_ERR_INVALID_ARG
    # bad options
    o = tbe.Options()
    lib.tbe_default_options(ctypes.byref(o))
    o.chunk = 0
    fake = ctypes.c_void_p(256)
    t2 = tbe.Tables(fake, fake, fake)
    assert lib.tbe_forward(ctypes.byref(p), ctypes.byref(o), ctypes.byref(t2), fake, fake, fake, None, fake,
                           None, 0, None, None) == tbe.TBE_ERR_INVALID_ARG
    # psw must be given exactly when the problem is weighted
    lib.tbe_default_options(ctypes.byref(o))
    assert lib.tbe_forward(ctypes.byref(p), ctypes.byref(o), ctypes.byref(t2), fake, fake, fake, fake, fake,
                           None, 0, None, None) == tbe.TBE_ERR_INVALID_ARG


def test_library_refuses_to_hide_a_missing_build(tmp_path):
    with pytest.raises(tbe.TBEError):
        tbe.load(str(tmp_path / "missing.so"))


def test_misaligned_buffers_are_rejected_on_the_host(lib):
    """Buffers the kernels read element by element must be aligned to their element (8 bytes for
    int64 indices, offsets, layout arrays and counters; 4 for fp32 arrays): a misaligned one is
    an argument error here rather than a fault on the device."""
    p, keep = _problem([8], [10])
    o = tbe.Options()
    lib.tbe_default_options(ctypes.byref(o))
    ok = ctypes.c_void_p(256)
    odd8, odd4 = ctypes.c_void_p(260), ctypes.c_void_p(258)
    t_ok = tbe.Tables(ok, ok, ok)
    for bad_tables in (tbe.Tables(odd8, ok, ok), tbe.Tables(ok, odd4, ok), tbe.Tables(ok, ok, odd8)):
        assert lib.tbe_forward(ctypes.byref(p), ctypes.byref(o), ctypes.byref(bad_tables), ok, ok, ok, None, ok,
                               None, 0, None, None) == tbe.TBE_ERR_INVALID_ARG
    # int64 indices / offsets at a 4-byte boundary
    assert lib.tbe_forward(ctypes.byref(p), ctypes.byref(o), ctypes.byref(t_ok), ok, odd8, ok, None, ok,
                           None, 0, None, None) == tbe.TBE_ERR_INVALID_ARG
    assert lib.tbe_bounds_check_offsets(ctypes.byref(p), ctypes.byref(t_ok), odd8, ok, 4096, None,
                                        None) == tbe.TBE_ERR_INVALID_ARG
    # the int64 counters
    assert lib.tbe_bounds_check(ctypes.byref(p), ctypes.byref(t_ok), ok, ok, ok, 4096, odd8,
                                None) == tbe.TBE_ERR_INVALID_ARG
    # the fp32 Adagrad state
    assert lib.tbe_backward_update(ctypes.byref(p), ctypes.byref(o), ctypes.byref(t_ok), ok, odd4, ok, ok, None,
                                   ok, tbe.TBE_OPT_ROWWISE_ADAGRAD, 0.1, 1e-8, ok, 1 << 30, None,
                                   None) == tbe.TBE_ERR_INVALID_ARG
    # int32 ids are fine at a 4-byte boundary but not at a 2-byte one
    p32, keep32 = _problem([8], [10], itype=tbe.TBE_I32)
    assert lib.tbe_forward(ctypes.byref(p32), ctypes.byref(o), ctypes.byref(t_ok), ok, ctypes.c_void_p(258), ok,
                           None, ok, None, 0, None, None) == tbe.TBE_ERR_INVALID_ARG


def test_checked_flavour_builds_with_the_same_exports():
    """The TBE_CHECKED debug library (device-side range checks counted in
    TBE_STAT_CHECK_FAILED) compiles from the same sources and exports the same C-ABI."""
    path = tbe_build.build(checked=True)
    assert path == tbe_build.CHECKED_LIB_PATH and path != tbe_build.LIB_PATH
    checked = tbe.load(path)
    for name in declared_functions():
        assert hasattr(checked, name), f"{name} missing from the checked library"
    assert tbe.STAT_NAMES[4] == "check_failed"


def test_forward_workspace_holds_the_saved_counts(lib):
    """tbe_forward_workspace_size(): 128 bytes per bag for each counts x table table (fp16,
    E <= 64, 64 <= D <= 128, long bags, unweighted sum pooling), at most 8 of them; 0 when no
    table qualifies or the path is off."""
    D = [128] * 10 + [64, 96]
    E = [64] * 10 + [1000, 50]
    flags = [1] * 10 + [1, 0]  # table 10 is too tall, table 11 has no long-bags flag
    long_bags = (ctypes.c_uint8 * len(D))(*flags)
    p, keep = _problem(D, E, B=100, n=1000)
    p.long_bags = ctypes.cast(long_bags, ctypes.POINTER(ctypes.c_uint8))
    o = tbe.Options()
    lib.tbe_default_options(ctypes.byref(o))
    assert lib.tbe_forward_workspace_size(ctypes.byref(p), ctypes.byref(o)) == 8 * 100 * 128
    o.histogram = 0
    assert lib.tbe_forward_workspace_size(ctypes.byref(p), ctypes.byref(o)) == 0
    lib.tbe_default_options(ctypes.byref(o))
    p.weighted = 1
    assert lib.tbe_forward_workspace_size(ctypes.byref(p), ctypes.byref(o)) == 0
    p.weighted = 0
    p.long_bags = None
    assert lib.tbe_forward_workspace_size(ctypes.byref(p), ctypes.byref(o)) == 0


def test_misaligned_forward_ws_is_rejected_on_the_host(lib):
    """tbe_options.forward_ws must be 16-byte aligned: the options are rejected (workspace queries
    answer 0, entry points INVALID_ARG) before any launch.  Data pointers are NULL, so that
    nothing could reach a kernel even if a check were missing."""
    p, keep = _problem([8], [10])
    t = tbe.Tables(None, None, None)
    o = tbe.Options()
    lib.tbe_default_options(ctypes.byref(o))
    o.forward_ws = 256 + 8
    assert lib.tbe_backward_workspace_size(ctypes.byref(p), ctypes.byref(o)) == 0
    assert lib.tbe_forward_workspace_size(ctypes.byref(p), ctypes.byref(o)) == 0
    assert lib.tbe_backward_update(ctypes.byref(p), ctypes.byref(o), ctypes.byref(t), None, None, None, None,
                                   None, None, tbe.TBE_OPT_ROWWISE_ADAGRAD, 0.1, 1e-8, None, 0, None,
                                   None) == tbe.TBE_ERR_INVALID_ARG
    o.forward_ws = 256
    assert lib.tbe_forward_workspace_size(ctypes.byref(p), ctypes.byref(o)) == 0  # no counts-path table
