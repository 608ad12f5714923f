"""The Python binding makes the tensors' device current around every library
call (the library launches on, and keeps its per-device state for, the current
device).  Checked on the CPU: the library and the device guard are replaced by
recorders and the tensors by metadata-only stand-ins on "cuda:1"; nothing is
launched anywhere."""
import contextlib

import pytest
import torch

import recurrent_state_02_gb300 as la
from recurrent_state_02_gb300 import _native

DEV = torch.device("cuda", 1)


class FakeTensor:
    """Metadata of a contiguous CUDA tensor; data_ptr is a dummy 16-byte-aligned value."""

    def __init__(self, shape, dtype, device=DEV):
        self.shape = tuple(shape)
        self.dtype = dtype
        self.device = device
        self.is_cuda = device.type == "cuda"

    def is_contiguous(self):
        return True

    def dim(self):
        return len(self.shape)

    def data_ptr(self):
        return 1 << 20

    def numel(self):
        n = 1
        for s in self.shape:
            n *= s
        return n

    def element_size(self):
        return {torch.bfloat16: 2, torch.float32: 4, torch.int32: 4, torch.uint8: 1}[self.dtype]


class Recorder:
    def __init__(self):
        self.current = None     # the device the guard made current
        self.calls = []         # (entry point, current device during the call)

    def guard(self, device):
        @contextlib.contextmanager
        def cm():
            prev, self.current = self.current, torch.device(device)
            try:
                yield
            finally:
                self.current = prev
        return cm()

    def lib(self):
        rec = self

        class Lib:
            def __getattr__(self, name):
                def fn(*args):
                    rec.calls.append((name, rec.current))
                    return 0
                return fn
        return Lib()


@pytest.fixture
def rec(monkeypatch):
    r = Recorder()
    monkeypatch.setattr(la, "_device_guard", r.guard)
    monkeypatch.setattr(la, "_stream", lambda device: 0)
    monkeypatch.setattr(_native, "lib", r.lib)
    return r


def _check(rec, *entries):
    seen = [name for name, _ in rec.calls]
    for e in entries:
        assert e in seen, (e, seen)
    for name, cur in rec.calls:
        if name in entries:
            assert cur == DEV, f"{name} was called with {cur} current, tensors on {DEV}"


def test_every_wrapper_calls_with_the_tensors_device_current(rec, monkeypatch):
    # outputs the wrappers allocate themselves become stand-ins on the same device
    monkeypatch.setattr(torch, "empty_like", lambda t: FakeTensor(t.shape, t.dtype, t.device))
    monkeypatch.setattr(torch, "empty", lambda shape, device=None, dtype=torch.float32:
                        FakeTensor(shape, dtype, torch.device(device)))
    B, H, T, r, dv = 2, 3, 70, 128, 128
    bf, f32 = torch.bfloat16, torch.float32
    q, k, v, y = (FakeTensor((B, H, T, n), bf) for n in (r, r, dv, dv))
    S, z = FakeTensor((B, H, r, dv), f32), FakeTensor((B, H, r), f32)
    alpha = FakeTensor((B, H, T), f32)

    la.state_init(B, H, r, dv, S=S, z=z)
    la.prefill_chunked(q, k, v, alpha=alpha, S0=S, z0=z, y=y, S_out=S, z_out=z)
    la.prefill_chunked_noalloc(q, k, v, y, S, z, alpha=alpha)
    qd, kd, vd, yd = (FakeTensor((B, H, 1, n), bf) for n in (r, r, dv, dv))
    la.decode_step(qd, kd, vd, S, z, y=yd)
    tq, tk, tv = (FakeTensor((T, H, n), bf) for n in (r, r, dv))
    cu = FakeTensor((B + 1,), torch.int32)
    la.prefill_varlen(tq, tk, tv, cu, y=FakeTensor((T, H, dv), bf), S_out=S, z_out=z)
    la.delta_rule(q, k, v, y=y, S_out=S)
    la.delta_rule_chunked(q, k, v, y=y, S_out=S, workspace=FakeTensor((1 << 20,), torch.uint8))
    la.prefill_backward(q, k, v, y, y, alpha=alpha, workspace=FakeTensor((1 << 20,), torch.uint8))
    la.prefill_chunked(q, k, v)   # outputs allocated by the wrapper
    la.last_device_status(DEV)
    _check(rec, "la_state_init", "la_prefill_chunked", "la_prefill_workspace_bytes", "la_prefill_chunked_noalloc",
           "la_decode_step", "la_prefill_varlen_workspace_bytes", "la_prefill_varlen", "la_delta_rule", "la_delta_rule_chunked", "la_prefill_backward", "la_last_device_status")


def test_tensors_on_another_device_are_refused(rec):
    q = FakeTensor((1, 1, 4, 128), torch.bfloat16)
    k = FakeTensor((1, 1, 4, 128), torch.bfloat16, device=torch.device("cuda", 0))
    with pytest.raises(ValueError):
        la.prefill_chunked(q, k, q)
    assert rec.calls == []
