"""The C-ABI library loads, exports every symbol include/linattn.h declares, and
rejects bad arguments on the host (these calls return before any CUDA work, so
they run without a GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "linattn.h")


@pytest.fixture(scope="module")
def native():
    from recurrent_state_02_gb300 import build, _native
    build.build()
    return _native


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(la_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("la_state_init", "la_prefill_chunked", "la_decode_step", "la_prefill_workspace_bytes",
                     "la_last_device_status", "la_status_string"):
        assert required in names


def test_every_declared_symbol_is_exported(native):
    lib = ctypes.CDLL(native.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(declared_functions()) == set(native.SIGNATURES), "binding and header disagree"


def test_status_strings(native):
    for code in range(9):
        s = native.status_string(code)
        assert s.startswith("LA_")
    assert native.status_string(99) == "unknown la_status"


def test_workspace_query(native):
    assert native.lib().la_prefill_workspace_bytes(4, 16, 4096, 128, 128, 64) == 0
    assert native.lib().la_prefill_workspace_bytes(4, 16, 4096, 128, 128, 0) == 0


FAKE = 1 << 20  # a 16-byte aligned non-null address; never dereferenced (validation fails first)


def _prefill(native, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, dtype=native.LA_DTYPE_BF16, alpha=None, S0=None, z0=None, B=1, H=1, T=64,
             r=128, dv=128, chunk=64, eps=1e-6, y=FAKE, S_out=FAKE, z_out=FAKE, ws=None, ws_bytes=0, stream=None)
    a.update(kw)
    return native.lib().la_prefill_chunked(a["q"], a["k"], a["v"], a["dtype"], a["alpha"], a["S0"], a["z0"],
                                           a["B"], a["H"], a["T"], a["r"], a["dv"], a["chunk"], a["eps"], a["y"],
                                           a["S_out"], a["z_out"], a["ws"], a["ws_bytes"], a["stream"])


def test_prefill_rejects_bad_arguments(native):
    """LC input contract (empty sequence, mismatched widths) as status codes."""
    assert _prefill(native, q=None) == native.LA_ERR_NULL
    assert _prefill(native, y=None) == native.LA_ERR_NULL
    assert _prefill(native, z_out=None) == native.LA_ERR_NULL
    assert _prefill(native, T=0) == native.LA_ERR_SHAPE
    assert _prefill(native, B=0) == native.LA_ERR_SHAPE
    assert _prefill(native, H=-1) == native.LA_ERR_SHAPE
    assert _prefill(native, r=0) == native.LA_ERR_SHAPE
    assert _prefill(native, chunk=0) == native.LA_ERR_SHAPE
    assert _prefill(native, dtype=7) == native.LA_ERR_DTYPE
    assert _prefill(native, r=64) == native.LA_ERR_UNSUPPORTED
    assert _prefill(native, dv=96) == native.LA_ERR_UNSUPPORTED
    # any chunk length >= 1 is accepted on BF16 (computed in chunks of 64; the result
    # does not depend on it): validation passes it on to the alignment checks
    assert _prefill(native, chunk=32, q=FAKE + 2) == native.LA_ERR_ALIGN
    assert _prefill(native, chunk=1000, q=FAKE + 2) == native.LA_ERR_ALIGN
    assert _prefill(native, q=FAKE + 2) == native.LA_ERR_ALIGN
    assert _prefill(native, y=FAKE + 8) == native.LA_ERR_ALIGN
    assert _prefill(native, alpha=FAKE + 1) == native.LA_ERR_ALIGN
    assert _prefill(native, dtype=native.LA_DTYPE_FP32, r=257) == native.LA_ERR_UNSUPPORTED
    assert _prefill(native, dtype=native.LA_DTYPE_FP32, dv=300) == native.LA_ERR_UNSUPPORTED
    assert _prefill(native, dtype=native.LA_DTYPE_FP32, q=FAKE + 2) == native.LA_ERR_ALIGN


def test_decode_rejects_bad_arguments(native):
    L = native.lib()
    f = lambda **kw: L.la_decode_step(kw.get("q", FAKE), FAKE, FAKE, kw.get("dtype", 0), None, kw.get("S", FAKE),
                                      FAKE, kw.get("B", 4), 2, kw.get("r", 128), kw.get("dv", 128), 1e-6, FAKE, None)
    assert f(q=None) == native.LA_ERR_NULL
    assert f(S=None) == native.LA_ERR_NULL
    assert f(B=0) == native.LA_ERR_SHAPE
    assert f(dtype=5) == native.LA_ERR_DTYPE
    assert f(r=257) == native.LA_ERR_UNSUPPORTED
    assert f(q=FAKE + 1) == native.LA_ERR_ALIGN
    assert f(S=FAKE + 2) == native.LA_ERR_ALIGN
    assert f(B=1 << 30) == native.LA_ERR_SHAPE   # B * H = 2^31 CTAs exceed the grid


def test_state_init_rejects_bad_arguments(native):
    L = native.lib()
    assert L.la_state_init(None, FAKE, 1, 1, 1, 1, None) == native.LA_ERR_NULL
    assert L.la_state_init(FAKE, FAKE, 1, 0, 1, 1, None) == native.LA_ERR_SHAPE
    assert L.la_state_init(FAKE + 1, FAKE, 1, 1, 1, 1, None) == native.LA_ERR_ALIGN
    assert L.la_debug_wait_probe(2_000_000_000, None) == native.LA_ERR_SHAPE


def test_workloads_follow_the_recipe():
    """The seeded generators: shapes, dtypes, gate range, determinism."""
    import torch
    from recurrent_state_02_gb300 import workloads as W
    w = W.GATED.with_(T=300)
    a = W.prefill_inputs(w)
    b = W.prefill_inputs(w)
    assert torch.equal(a["q"], b["q"]) and torch.equal(a["alpha"], b["alpha"])
    assert a["q"].dtype == torch.bfloat16 and a["q"].shape == (2, 16, 300, 128)
    assert a["alpha"].dtype == torch.float32 and float(a["alpha"].min()) > 0 and float(a["alpha"].max()) < 1
    assert abs(float(a["alpha"].mean()) - 0.93) < 0.03  # sigmoid(N(3,1)) has mean ~0.93
    d = W.decode_inputs(W.DECODE.with_(B=8))
    assert d["S"].shape == (8, 16, 128, 128) and float(d["z"].min()) >= 1 and float(d["z"].max()) <= 100
    t = W.prefill_inputs(W.TINY)
    assert t["q"].dtype == torch.float32 and t["q"].shape == (1, 1, 64, 16)
    assert W.LONG.scale == 2.0 and W.UNGATED.chunk == 64


def _varlen(native, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, dtype=native.LA_DTYPE_BF16, alpha=None, S0=None, z0=None, cu=FAKE, B=2, H=1,
             T=100, r=128, dv=128, chunk=64, eps=1e-6, y=FAKE, S_out=FAKE, z_out=FAKE, ws=None, ws_bytes=0,
             stream=None)
    a.update(kw)
    return native.lib().la_prefill_varlen(a["q"], a["k"], a["v"], a["dtype"], a["alpha"], a["S0"], a["z0"], a["cu"],
                                          a["B"], a["H"], a["T"], a["r"], a["dv"], a["chunk"], a["eps"], a["y"],
                                          a["S_out"], a["z_out"], a["ws"], a["ws_bytes"], a["stream"])


def test_varlen_rejects_bad_arguments(native):
    assert _varlen(native, cu=None) == native.LA_ERR_NULL
    assert _varlen(native, q=None) == native.LA_ERR_NULL
    assert _varlen(native, S_out=None) == native.LA_ERR_NULL
    assert _varlen(native, B=0) == native.LA_ERR_SHAPE
    assert _varlen(native, T=-1) == native.LA_ERR_SHAPE
    assert _varlen(native, dtype=9) == native.LA_ERR_DTYPE
    assert _varlen(native, dtype=native.LA_DTYPE_FP32) == native.LA_ERR_UNSUPPORTED
    assert _varlen(native, dv=96) == native.LA_ERR_UNSUPPORTED
    assert _varlen(native, q=FAKE + 8) == native.LA_ERR_ALIGN
    assert _varlen(native, cu=FAKE + 2) == native.LA_ERR_ALIGN


def test_varlen_workspace_bytes(native):
    L = native.lib()
    # sizes la_prefill_varlen rejects need nothing
    for args in ((0, 16, 4096, 128, 128), (4, 0, 4096, 128, 128), (4, 16, -1, 128, 128), (4, 16, 4096, 64, 128),
                 (4, 16, 4096, 128, 96)):
        assert L.la_prefill_varlen_workspace_bytes(*args) == 0
    # the plan follows the current device's SM count (none here): no segments
    assert L.la_prefill_varlen_workspace_bytes(48, 16, 40448, 128, 128) == 0


def test_delta_rejects_bad_arguments(native):
    L = native.lib()

    def f(**kw):
        a = dict(q=FAKE, k=FAKE, v=FAKE, dtype=native.LA_DTYPE_BF16, beta=None, S0=None, B=1, H=1, T=64, r=128,
                 dv=128, y=FAKE, S_out=FAKE)
        a.update(kw)
        return L.la_delta_rule(a["q"], a["k"], a["v"], a["dtype"], a["beta"], a["S0"], a["B"], a["H"], a["T"],
                               a["r"], a["dv"], a["y"], a["S_out"], None)

    assert f(q=None) == native.LA_ERR_NULL
    assert f(S_out=None) == native.LA_ERR_NULL
    assert f(T=0, S_out=None) == native.LA_ERR_NULL
    assert f(B=0) == native.LA_ERR_SHAPE
    assert f(T=-1) == native.LA_ERR_SHAPE
    assert f(dtype=4) == native.LA_ERR_DTYPE
    assert f(r=96) == native.LA_ERR_UNSUPPORTED
    assert f(dv=48) == native.LA_ERR_UNSUPPORTED
    assert f(v=FAKE + 8) == native.LA_ERR_ALIGN
    assert f(beta=FAKE + 2) == native.LA_ERR_ALIGN
    assert f(S0=FAKE + 4) == native.LA_ERR_ALIGN
    assert f(S_out=FAKE + 4) == native.LA_ERR_ALIGN


def test_delta_chunked_rejects_bad_arguments(native):
    L = native.lib()

    def f(**kw):
        a = dict(q=FAKE, k=FAKE, v=FAKE, dtype=native.LA_DTYPE_BF16, beta=None, S0=None, B=1, H=1, T=64, r=128,
                 dv=128, y=FAKE, S_out=FAKE, ws=FAKE, ws_bytes=32768)
        a.update(kw)
        return L.la_delta_rule_chunked(a["q"], a["k"], a["v"], a["dtype"], a["beta"], a["S0"], a["B"], a["H"],
                                       a["T"], a["r"], a["dv"], a["y"], a["S_out"], a["ws"], a["ws_bytes"], None)

    assert L.la_delta_chunked_workspace_bytes(4, 16, 4096) == 4 * 16 * 64 * 32768
    assert L.la_delta_chunked_workspace_bytes(1, 1, 65) == 2 * 32768
    assert L.la_delta_chunked_workspace_bytes(1, 1, 0) == 0

    assert f(k=None) == native.LA_ERR_NULL
    assert f(S_out=None) == native.LA_ERR_NULL
    assert f(H=0) == native.LA_ERR_SHAPE
    assert f(T=-1) == native.LA_ERR_SHAPE
    assert f(dtype=native.LA_DTYPE_FP32) == native.LA_ERR_DTYPE
    assert f(r=64) == native.LA_ERR_UNSUPPORTED
    assert f(dv=96) == native.LA_ERR_UNSUPPORTED
    assert f(y=FAKE + 8) == native.LA_ERR_ALIGN
    assert f(S0=FAKE + 8) == native.LA_ERR_ALIGN     # 16-byte alignment for the FP32 state here
    assert f(S_out=FAKE + 8) == native.LA_ERR_ALIGN
    assert f(beta=FAKE + 2) == native.LA_ERR_ALIGN
    assert f(ws=None) == native.LA_ERR_WORKSPACE
    assert f(ws_bytes=16383) == native.LA_ERR_WORKSPACE
    assert f(T=65) == native.LA_ERR_WORKSPACE           # two chunks need 32 KB
    assert f(ws=FAKE + 8) == native.LA_ERR_ALIGN


def test_saved_denominator_entries_reject_bad_arguments(native):
    """la_prefill_chunked_save needs d_out, 4-byte aligned; la_prefill_backward_saved
    needs d, 4-byte aligned; otherwise they check what their plain forms check."""
    L = native.lib()

    def fwd(**kw):
        a = dict(q=FAKE, dtype=native.LA_DTYPE_BF16, T=64, d_out=FAKE, y=FAKE)
        a.update(kw)
        return L.la_prefill_chunked_save(a["q"], FAKE, FAKE, a["dtype"], None, None, None, 1, 1, a["T"], 128, 128, 64,
                                         1e-6, a["y"], FAKE, FAKE, a["d_out"], a.get("states"), None, 0, None)

    assert fwd(d_out=None) == native.LA_ERR_NULL
    assert fwd(q=None) == native.LA_ERR_NULL
    assert fwd(T=0) == native.LA_ERR_SHAPE
    assert fwd(dtype=7) == native.LA_ERR_DTYPE
    assert fwd(d_out=FAKE + 2) == native.LA_ERR_ALIGN
    assert fwd(dtype=native.LA_DTYPE_FP32, d_out=FAKE + 2) == native.LA_ERR_ALIGN
    assert fwd(states=FAKE + 4) == native.LA_ERR_ALIGN

    def bwd(**kw):
        a = dict(q=FAKE, d=FAKE, T=64, ws=FAKE, ws_bytes=1 << 20)
        a.update(kw)
        return L.la_prefill_backward_saved(a["q"], FAKE, FAKE, native.LA_DTYPE_BF16, None, None, None, 1, 1, a["T"],
                                           128, 128, FAKE, FAKE, a["d"], a.get("states"), None, None, FAKE, FAKE,
                                           FAKE, None, FAKE, FAKE, a["ws"], a["ws_bytes"], None)

    assert bwd(d=None) == native.LA_ERR_NULL
    assert bwd(q=None) == native.LA_ERR_NULL
    assert bwd(T=0) == native.LA_ERR_SHAPE
    assert bwd(d=FAKE + 2) == native.LA_ERR_ALIGN
    assert bwd(ws=None) == native.LA_ERR_WORKSPACE
    assert bwd(states=FAKE + 4) == native.LA_ERR_ALIGN
    # without a device there are no SMs to fill, so no segments and nothing to keep
    assert L.la_backward_states_bytes(4, 16, 4096) == 0
    assert L.la_backward_states_bytes(0, 16, 4096) == 0


def test_backward_rejects_bad_arguments(native):
    L = native.lib()

    def f(**kw):
        a = dict(q=FAKE, dtype=native.LA_DTYPE_BF16, alpha=None, B=1, H=1, T=64, r=128, dv=128, y=FAKE, dS_T=None,
                 dalpha=None, dS0=FAKE, ws=FAKE, ws_bytes=1 << 20)
        a.update(kw)
        return L.la_prefill_backward(a["q"], FAKE, FAKE, a["dtype"], a["alpha"], None, None, a["B"], a["H"], a["T"],
                                     a["r"], a["dv"], 1e-6, a["y"], FAKE, a["dS_T"], None, FAKE, FAKE, FAKE,
                                     a["dalpha"], a["dS0"], FAKE, a["ws"], a["ws_bytes"], None)

    assert f(q=None) == native.LA_ERR_NULL
    assert f(dS0=None) == native.LA_ERR_NULL
    assert f(T=0) == native.LA_ERR_SHAPE
    assert f(dtype=3) == native.LA_ERR_DTYPE
    assert f(r=96) == native.LA_ERR_UNSUPPORTED
    assert f(dv=256) == native.LA_ERR_UNSUPPORTED
    assert f(y=FAKE + 1) == native.LA_ERR_ALIGN
    assert f(dS_T=FAKE + 4) == native.LA_ERR_ALIGN
    assert f(ws=None) == native.LA_ERR_WORKSPACE
    assert f(ws_bytes=16) == native.LA_ERR_WORKSPACE
    # d, dd, the dalpha terms [B*H*T] and fin [B*H], then the z pass's maps (P, zs and
    # z_start per 128-token segment, r <= 128), rounded up to 256 bytes; without a
    # device (no SMs) there are no sequence segments and no state-pass workspace
    BH, T = 4 * 16, 4096
    nzs = (T + 127) // 128
    floats = BH * (3 * T + 1) + BH * nzs * (1 + 2 * 128) + 4
    assert L.la_backward_workspace_bytes(4, 16, 4096) == (4 * floats + 255) // 256 * 256
