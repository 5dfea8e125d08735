"""The Python binding calls every library entry point with the problem's device current and on
that device's stream (or the stream the caller passes): the library launches on the current
device, so a call made while another device is current must not reach it there.  Host logic
only: the library and the CUDA device context are fakes, and no GPU is needed."""
import types

import pytest
import torch

from bwd_tbe_fwd_gb300 import tbe

DEV = torch.device("cpu")  # the fakes below stand in for the CUDA device context


class FakeDeviceContext:
    """Replaces torch.cuda.device: records which device is current while the library runs."""
    current = "other"

    def __init__(self, device):
        self.device = device

    def __enter__(self):
        self.prev = FakeDeviceContext.current
        FakeDeviceContext.current = self.device
        return self

    def __exit__(self, *exc):
        FakeDeviceContext.current = self.prev
        return False


def fake_stream_of(device):
    return types.SimpleNamespace(cuda_stream=1000 if device == DEV else 2000)


class FakeLib:
    """Each entry point records (its name, the current device, its stream argument) and returns OK."""

    def __init__(self):
        self.calls = []

    def _entry(self, name):
        def fn(*args):
            self.calls.append((name, FakeDeviceContext.current, args[-1].value))
            return tbe.TBE_OK
        return fn

    def __getattr__(self, name):
        if not name.startswith("tbe_"):
            raise AttributeError(name)
        fn = self._entry(name)
        setattr(self, name, fn)
        return fn


@pytest.fixture
def emb(monkeypatch):
    monkeypatch.setattr(torch.cuda, "device", FakeDeviceContext)
    monkeypatch.setattr(torch.cuda, "current_stream", lambda device=None: fake_stream_of(device))
    e = tbe.TableBatchedEmbedding.__new__(tbe.TableBatchedEmbedding)
    e.lib = FakeLib()
    e.device = DEV
    e.D, e.E, e.T, e.B = [8, 4], [10, 6], 2, 3
    e.num_indices = 12
    e.weight_dtype, e.index_dtype = torch.float16, torch.int64
    e.weighted = True
    e.prob = tbe.Problem()
    e.tables = tbe.Tables()
    e.options = tbe.TBEOptions()
    e.num_weights, e.total_rows, e.total_D = 8 * 10 + 4 * 6, 16, 12
    e.ws_bounds = torch.empty(256, dtype=torch.uint8)
    e.ws_forward = torch.empty(256, dtype=torch.uint8)
    e.ws_backward = torch.empty(256, dtype=torch.uint8)
    return e


def _inputs(e):
    return dict(
        weights=torch.zeros(e.num_weights, dtype=torch.float16),
        indices=torch.zeros(e.num_indices, dtype=torch.int64),
        offsets=torch.zeros(e.T * e.B + 1, dtype=torch.int64),
        psw=torch.ones(e.num_indices, dtype=torch.float32),
        grad=torch.zeros(e.B, e.total_D, dtype=torch.float32),
        state=torch.zeros(e.total_rows, dtype=torch.float32),
    )


def _run_all(e, stream):
    x = _inputs(e)
    e.bounds_check(x["indices"], x["offsets"], stream=stream)
    e.bounds_check(x["indices"], x["offsets"], stream=stream, offsets_only=True)
    e.forward(x["weights"], x["indices"], x["offsets"], psw=x["psw"], stream=stream)
    e.psw_gradient(x["weights"], x["indices"], x["offsets"], x["grad"], stream=stream)
    e.backward_prepare(x["indices"], x["offsets"], psw=x["psw"], stream=stream)
    e.backward_update(x["weights"], x["state"], x["indices"], x["offsets"], x["grad"], psw=x["psw"],
                      stream=stream, prepared=True)
    tbe.tbe_backward_update_noalloc(e, x["weights"], x["state"], x["indices"], x["offsets"], x["grad"],
                                    psw=x["psw"], stream=stream)


def test_every_call_runs_on_the_problems_device_and_stream(emb):
    _run_all(emb, stream=None)
    names = [c[0] for c in emb.lib.calls]
    assert names == ["tbe_bounds_check", "tbe_bounds_check_offsets", "tbe_forward", "tbe_psw_gradient",
                     "tbe_backward_prepare", "tbe_backward_update", "tbe_backward_update_noalloc"]
    for name, dev, stream in emb.lib.calls:
        assert dev == DEV, f"{name} ran with {dev!r} current"
        assert stream == 1000, f"{name} did not take the problem device's current stream"
    assert FakeDeviceContext.current == "other"  # the caller's device is current again


def test_an_explicit_stream_is_passed_through(emb):
    mine = types.SimpleNamespace(cuda_stream=4242)
    _run_all(emb, stream=mine)
    assert all(dev == DEV and stream == 4242 for _, dev, stream in emb.lib.calls)

