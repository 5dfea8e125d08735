"""The give-up path of the library's bounded device waits ("Modernizing Table Batched Embeddings
with FBTriton", section 4, Problem 5: no block may wait on another; the library bounds every wait
it has).  A CTA waits on an mbarrier phase that nothing completes; after a few polls it must count
TBE_STAT_WAIT_TIMEOUT and return, leaving the context usable for the next launch."""
import ctypes

import pytest
import torch

from bwd_tbe_fwd_gb300 import tbe

pytestmark = pytest.mark.gpu

TBE_STAT_WAIT_TIMEOUT = 3


def test_bounded_wait_gives_up_and_counts():
    stats = torch.zeros(tbe.TBE_NUM_STATS, dtype=torch.int64, device="cuda")
    tbe.selftest_wait_timeout(stats, polls=4)
    torch.cuda.synchronize()
    assert stats[TBE_STAT_WAIT_TIMEOUT].item() == 1
    assert stats.sum().item() == 1  # nothing else counted
    tbe.selftest_wait_timeout(stats, polls=64)
    torch.cuda.synchronize()
    assert stats[TBE_STAT_WAIT_TIMEOUT].item() == 2
    # the context still runs work after the give-ups
    x = torch.arange(1024, device="cuda", dtype=torch.float32)
    assert x.sum().item() == 1023 * 1024 / 2


def test_selftest_rejects_bad_arguments():
    lib = tbe.load()
    fn = lib.tbe_selftest_wait_timeout
    fn.argtypes = [ctypes.c_uint32, ctypes.c_void_p, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    stats = torch.zeros(tbe.TBE_NUM_STATS, dtype=torch.int64, device="cuda")
    assert fn(4, None, None) == tbe.TBE_ERR_INVALID_ARG
    assert fn(0, ctypes.c_void_p(stats.data_ptr()), None) == tbe.TBE_ERR_INVALID_ARG
    assert fn(5000, ctypes.c_void_p(stats.data_ptr()), None) == tbe.TBE_ERR_INVALID_ARG
    assert fn(4, ctypes.c_void_p(stats.data_ptr() + 4), None) == tbe.TBE_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert stats.sum().item() == 0
