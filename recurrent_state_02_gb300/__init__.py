"""GB300 (sm_103a) normalised causal linear attention with a recurrent S/z state.

    phi(x) = ELU(x) + 1
    S_t = alpha_t S_{t-1} + phi(k_t) v_t^T,   z_t = alpha_t z_{t-1} + phi(k_t)
    y_t = phi(q_t)^T S_t / (phi(q_t)^T z_t + eps)

Every step runs in the CUDA kernels of liblinattn.so, reached through its C ABI
(include/linattn.h).  The functions below only check tensor metadata, allocate
outputs with torch, and pass raw device pointers and the current CUDA stream;
PyTorch supplies device memory and streams, nothing else.
"""
from __future__ import annotations

import torch

from . import _native
from ._native import LinAttnError  # noqa: F401

_DTYPES = {torch.bfloat16: _native.LA_DTYPE_BF16, torch.float32: _native.LA_DTYPE_FP32}


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(device):
    return torch.cuda.current_stream(device).cuda_stream


def _device_guard(device):
    """Makes `device` current for the duration of a library call.  The library
    launches on the current device (the default stream's handle 0 names that
    device's stream) and keeps its per-device state (status word, scratch, SM
    count) for the current device, so the tensors' device must be current."""
    return torch.cuda.device(device)


def _require(t, name, shape, dtype, device):
    if t is None:
        return
    if not t.is_cuda or t.device != device:
        raise ValueError(f"{name} must be on {device}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.dtype != dtype:
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def state_init(B, H, r, dv, device="cuda", S=None, z=None):
    """Zero state: returns (S [B,H,r,dv], z [B,H,r]) in FP32."""
    device = torch.device(device)
    if S is None:
        S = torch.empty((B, H, r, dv), device=device, dtype=torch.float32)
    if z is None:
        z = torch.empty((B, H, r), device=device, dtype=torch.float32)
    _require(S, "S", (B, H, r, dv), torch.float32, S.device)
    _require(z, "z", (B, H, r), torch.float32, S.device)
    with _device_guard(S.device):
        st = _native.lib().la_state_init(_ptr(S), _ptr(z), B, H, r, dv, _stream(S.device))
    _native.check(st, "la_state_init")
    return S, z


def prefill_workspace_bytes(B, H, T, r, dv, chunk=64, device=None) -> int:
    """Scratch bytes of prefill_chunked for these sizes on `device` (default: the
    current device); the plan depends on the device's SM count."""
    if device is None:
        return int(_native.lib().la_prefill_workspace_bytes(B, H, T, r, dv, chunk))
    with _device_guard(torch.device(device)):
        return int(_native.lib().la_prefill_workspace_bytes(B, H, T, r, dv, chunk))


def prefill_chunked(q, k, v, alpha=None, S0=None, z0=None, chunk=64, eps=1e-6, y=None, S_out=None, z_out=None,
                    workspace=None):
    """Chunkwise prefill.  q, k [B,H,T,r], v [B,H,T,dv] (bf16 or fp32, same dtype);
    alpha [B,H,T] fp32 or None; S0 [B,H,r,dv], z0 [B,H,r] fp32 or None.
    Returns (y [B,H,T,dv] in the input dtype, S_T, z_T)."""
    return _prefill(q, k, v, alpha, S0, z0, chunk, eps, y, S_out, z_out, workspace, None)


def backward_states_bytes(B, H, T, device=None) -> int:
    """Bytes of the states a training forward can keep for the backward's sequence
    segments on `device` (0: the backward would not split the sequence)."""
    if device is None:
        return int(_native.lib().la_backward_states_bytes(B, H, T))
    with _device_guard(torch.device(device)):
        return int(_native.lib().la_backward_states_bytes(B, H, T))


def prefill_chunked_save(q, k, v, alpha=None, S0=None, z0=None, chunk=64, eps=1e-6, y=None, S_out=None, z_out=None,
                         d_out=None, workspace=None, keep_states=True):
    """prefill_chunked that also returns what the backward can reuse: d [B,H,T]
    fp32, the denominator of every output row (phi(q_t) . z_t + eps), and the
    states entering the backward's sequence segments (a flat fp32 tensor, or None
    when there are none or keep_states is False), for
    prefill_backward(..., d=d, states=states).  Returns (y, S_T, z_T, d, states)."""
    B, H, T, _ = q.shape
    if d_out is None:
        d_out = torch.empty((B, H, T), device=q.device, dtype=torch.float32)
    _require(d_out, "d_out", (B, H, T), torch.float32, q.device)
    states = None
    if keep_states and q.dtype == torch.bfloat16:
        nbytes = backward_states_bytes(B, H, T, device=q.device)
        if nbytes:
            states = torch.empty(nbytes // 4, device=q.device, dtype=torch.float32)
    return _prefill(q, k, v, alpha, S0, z0, chunk, eps, y, S_out, z_out, workspace, d_out, states) + (d_out, states)


def _prefill(q, k, v, alpha, S0, z0, chunk, eps, y, S_out, z_out, workspace, d_out, states=None):
    if q.dtype not in _DTYPES:
        raise ValueError(f"unsupported dtype {q.dtype}")
    B, H, T, r = q.shape
    dv = v.shape[3]
    dev = q.device
    _require(q, "q", (B, H, T, r), q.dtype, dev)
    _require(k, "k", (B, H, T, r), q.dtype, dev)
    _require(v, "v", (B, H, T, dv), q.dtype, dev)
    _require(alpha, "alpha", (B, H, T), torch.float32, dev)
    _require(S0, "S0", (B, H, r, dv), torch.float32, dev)
    _require(z0, "z0", (B, H, r), torch.float32, dev)
    if y is None:
        y = torch.empty((B, H, T, dv), device=dev, dtype=q.dtype)
    if S_out is None:
        S_out = torch.empty((B, H, r, dv), device=dev, dtype=torch.float32)
    if z_out is None:
        z_out = torch.empty((B, H, r), device=dev, dtype=torch.float32)
    _require(y, "y", (B, H, T, dv), q.dtype, dev)
    _require(S_out, "S_out", (B, H, r, dv), torch.float32, dev)
    _require(z_out, "z_out", (B, H, r), torch.float32, dev)
    need = prefill_workspace_bytes(B, H, T, r, dv, chunk, device=dev)
    if need and workspace is None:
        workspace = torch.empty(need, device=dev, dtype=torch.uint8)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    with _device_guard(dev):
        if d_out is None:
            st = _native.lib().la_prefill_chunked(
                _ptr(q), _ptr(k), _ptr(v), _DTYPES[q.dtype], _ptr(alpha), _ptr(S0), _ptr(z0), B, H, T, r, dv, chunk,
                float(eps), _ptr(y), _ptr(S_out), _ptr(z_out), _ptr(workspace), ws_bytes, _stream(dev))
            _native.check(st, "la_prefill_chunked")
        else:
            st = _native.lib().la_prefill_chunked_save(
                _ptr(q), _ptr(k), _ptr(v), _DTYPES[q.dtype], _ptr(alpha), _ptr(S0), _ptr(z0), B, H, T, r, dv, chunk,
                float(eps), _ptr(y), _ptr(S_out), _ptr(z_out), _ptr(d_out), _ptr(states), _ptr(workspace), ws_bytes,
                _stream(dev))
            _native.check(st, "la_prefill_chunked_save")
    return y, S_out, z_out


def varlen_workspace_bytes(B, H, total_T, r, dv, device=None) -> int:
    """Scratch bytes of prefill_varlen for these sizes on `device` (default: the
    current device); it depends on the device's SM count, not on the lengths."""
    if device is None:
        return int(_native.lib().la_prefill_varlen_workspace_bytes(B, H, total_T, r, dv))
    with _device_guard(torch.device(device)):
        return int(_native.lib().la_prefill_varlen_workspace_bytes(B, H, total_T, r, dv))


def prefill_varlen(q, k, v, cu_seqlens, alpha=None, S0=None, z0=None, chunk=64, eps=1e-6, y=None, S_out=None,
                   z_out=None, workspace=None):
    """Packed sequences of different lengths: q, k [total_T, H, r], v [total_T, H, dv]
    (bf16, token-major); cu_seqlens int32 [B+1] on the device (sequence b is tokens
    cu_seqlens[b] .. cu_seqlens[b+1]-1); alpha [total_T, H] fp32 or None; S0
    [B,H,r,dv], z0 [B,H,r] fp32 or None; workspace uint8 of varlen_workspace_bytes
    (allocated here when None).  Returns (y [total_T, H, dv], S_T, z_T)."""
    if q.dtype not in _DTYPES:
        raise ValueError(f"unsupported dtype {q.dtype}")
    total_T, H, r = q.shape
    dv = v.shape[2]
    dev = q.device
    if cu_seqlens.dtype != torch.int32 or cu_seqlens.dim() != 1 or cu_seqlens.device != dev:
        raise ValueError("cu_seqlens must be a 1-D int32 tensor on the device of q")
    B = cu_seqlens.numel() - 1
    _require(q, "q", (total_T, H, r), q.dtype, dev)
    _require(k, "k", (total_T, H, r), q.dtype, dev)
    _require(v, "v", (total_T, H, dv), q.dtype, dev)
    _require(cu_seqlens, "cu_seqlens", (B + 1,), torch.int32, dev)
    _require(alpha, "alpha", (total_T, H), torch.float32, dev)
    _require(S0, "S0", (B, H, r, dv), torch.float32, dev)
    _require(z0, "z0", (B, H, r), torch.float32, dev)
    if y is None:
        y = torch.empty((total_T, H, dv), device=dev, dtype=q.dtype)
    if S_out is None:
        S_out = torch.empty((B, H, r, dv), device=dev, dtype=torch.float32)
    if z_out is None:
        z_out = torch.empty((B, H, r), device=dev, dtype=torch.float32)
    _require(y, "y", (total_T, H, dv), q.dtype, dev)
    _require(S_out, "S_out", (B, H, r, dv), torch.float32, dev)
    _require(z_out, "z_out", (B, H, r), torch.float32, dev)
    need = varlen_workspace_bytes(B, H, total_T, r, dv, device=dev)
    if need and workspace is None:
        workspace = torch.empty(need, device=dev, dtype=torch.uint8)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    with _device_guard(dev):
        st = _native.lib().la_prefill_varlen(
            _ptr(q), _ptr(k), _ptr(v), _DTYPES[q.dtype], _ptr(alpha), _ptr(S0), _ptr(z0), _ptr(cu_seqlens), B, H,
            total_T, r, dv, chunk, float(eps), _ptr(y), _ptr(S_out), _ptr(z_out), _ptr(workspace), ws_bytes,
            _stream(dev))
    _native.check(st, "la_prefill_varlen")
    return y, S_out, z_out


def prefill_chunked_noalloc(q, k, v, y, S_out, z_out, alpha=None, S0=None, z0=None, chunk=64, eps=1e-6):
    """As prefill_chunked, with the library's built-in scratch instead of a
    workspace; nothing is allocated here either, so y [B,H,T,dv] (input dtype),
    S_out [B,H,r,dv] and z_out [B,H,r] (fp32) must be given.  Calls that may
    overlap in time share one buffer per device and must be serialised."""
    if q.dtype not in _DTYPES:
        raise ValueError(f"unsupported dtype {q.dtype}")
    B, H, T, r = q.shape
    dv = v.shape[3]
    dev = q.device
    _require(q, "q", (B, H, T, r), q.dtype, dev)
    _require(k, "k", (B, H, T, r), q.dtype, dev)
    _require(v, "v", (B, H, T, dv), q.dtype, dev)
    _require(alpha, "alpha", (B, H, T), torch.float32, dev)
    _require(S0, "S0", (B, H, r, dv), torch.float32, dev)
    _require(z0, "z0", (B, H, r), torch.float32, dev)
    if y is None or S_out is None or z_out is None:
        raise ValueError("y, S_out and z_out must be given (this entry point allocates nothing)")
    _require(y, "y", (B, H, T, dv), q.dtype, dev)
    _require(S_out, "S_out", (B, H, r, dv), torch.float32, dev)
    _require(z_out, "z_out", (B, H, r), torch.float32, dev)
    with _device_guard(dev):
        st = _native.lib().la_prefill_chunked_noalloc(
            _ptr(q), _ptr(k), _ptr(v), _DTYPES[q.dtype], _ptr(alpha), _ptr(S0), _ptr(z0), B, H, T, r, dv, chunk,
            float(eps), _ptr(y), _ptr(S_out), _ptr(z_out), _stream(dev))
    _native.check(st, "la_prefill_chunked_noalloc")
    return y, S_out, z_out


def decode_step(q, k, v, S, z, alpha=None, eps=1e-6, y=None):
    """One token per request, state updated in place.  q, k [B,H,1,r], v [B,H,1,dv];
    S [B,H,r,dv], z [B,H,r] fp32 (overwritten); alpha [B,H] fp32 or None.  Returns y [B,H,1,dv]."""
    if q.dtype not in _DTYPES:
        raise ValueError(f"unsupported dtype {q.dtype}")
    B, H, one, r = q.shape
    dv = v.shape[3]
    dev = q.device
    if one != 1:
        raise ValueError("decode takes one token per request")
    _require(k, "k", (B, H, 1, r), q.dtype, dev)
    _require(v, "v", (B, H, 1, dv), q.dtype, dev)
    _require(S, "S", (B, H, r, dv), torch.float32, dev)
    _require(z, "z", (B, H, r), torch.float32, dev)
    _require(alpha, "alpha", (B, H), torch.float32, dev)
    if y is None:
        y = torch.empty((B, H, 1, dv), device=dev, dtype=q.dtype)
    _require(y, "y", (B, H, 1, dv), q.dtype, dev)
    with _device_guard(dev):
        st = _native.lib().la_decode_step(_ptr(q), _ptr(k), _ptr(v), _DTYPES[q.dtype], _ptr(alpha), _ptr(S), _ptr(z),
                                          B, H, r, dv, float(eps), _ptr(y), _stream(dev))
    _native.check(st, "la_decode_step")
    return y


def prefill_backward(q, k, v, y, dy, alpha=None, S0=None, z0=None, dS_T=None, dz_T=None, eps=1e-6, workspace=None,
                     d=None, states=None):
    """Gradients of prefill_chunked: given the forward inputs, its output y and
    dy [B,H,T,dv] (and optionally dS_T [B,H,r,dv], dz_T [B,H,r] in fp32), returns
    (dq, dk, dv, dalpha or None, dS0, dz0); dq, dk, dv in the input dtype.
    d: the [B,H,T] fp32 denominators from prefill_chunked_save (eps is then not
    used), or None to recompute them; states: the segment states from the same
    call (with d only), or None."""
    if states is not None and d is None:
        raise ValueError("states are taken only together with d")
    if q.dtype not in _DTYPES:
        raise ValueError(f"unsupported dtype {q.dtype}")
    B, H, T, r = q.shape
    dvd = v.shape[3]
    dev = q.device
    for t, name, shape in ((q, "q", (B, H, T, r)), (k, "k", (B, H, T, r)), (v, "v", (B, H, T, dvd)),
                           (y, "y", (B, H, T, dvd)), (dy, "dy", (B, H, T, dvd))):
        _require(t, name, shape, q.dtype, dev)
    _require(alpha, "alpha", (B, H, T), torch.float32, dev)
    _require(S0, "S0", (B, H, r, dvd), torch.float32, dev)
    _require(z0, "z0", (B, H, r), torch.float32, dev)
    _require(dS_T, "dS_T", (B, H, r, dvd), torch.float32, dev)
    _require(dz_T, "dz_T", (B, H, r), torch.float32, dev)
    _require(d, "d", (B, H, T), torch.float32, dev)
    dq, dk, dv_out = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dalpha = torch.empty((B, H, T), device=dev, dtype=torch.float32) if alpha is not None else None
    dS0 = torch.empty((B, H, r, dvd), device=dev, dtype=torch.float32)
    dz0 = torch.empty((B, H, r), device=dev, dtype=torch.float32)
    need = int(_native.lib().la_backward_workspace_bytes(B, H, T))
    if workspace is None:
        workspace = torch.empty(need, device=dev, dtype=torch.uint8)
    ws_bytes = workspace.numel() * workspace.element_size()
    with _device_guard(dev):
        if d is None:
            st = _native.lib().la_prefill_backward(
                _ptr(q), _ptr(k), _ptr(v), _DTYPES[q.dtype], _ptr(alpha), _ptr(S0), _ptr(z0), B, H, T, r, dvd,
                float(eps), _ptr(y), _ptr(dy), _ptr(dS_T), _ptr(dz_T), _ptr(dq), _ptr(dk), _ptr(dv_out), _ptr(dalpha),
                _ptr(dS0), _ptr(dz0), _ptr(workspace), ws_bytes, _stream(dev))
            _native.check(st, "la_prefill_backward")
        else:
            st = _native.lib().la_prefill_backward_saved(
                _ptr(q), _ptr(k), _ptr(v), _DTYPES[q.dtype], _ptr(alpha), _ptr(S0), _ptr(z0), B, H, T, r, dvd,
                _ptr(y), _ptr(dy), _ptr(d), _ptr(states), _ptr(dS_T), _ptr(dz_T), _ptr(dq), _ptr(dk), _ptr(dv_out),
                _ptr(dalpha), _ptr(dS0), _ptr(dz0), _ptr(workspace), ws_bytes, _stream(dev))
            _native.check(st, "la_prefill_backward_saved")
    return dq, dk, dv_out, dalpha, dS0, dz0


def delta_rule(q, k, v, beta=None, S0=None, y=None, S_out=None):
    """Delta-rule memory: p = S^T k, S += beta k (v - p)^T, y = S^T q (after the write).
    q, k [B,H,T,r], v [B,H,T,dv] (bf16 or fp32, same dtype); beta [B,H,T] fp32 or
    None (1); S0 [B,H,r,dv] fp32 or None (zero).  Returns (y [B,H,T,dv], S_T).
    The token recurrence in FP32 (la_delta_rule)."""
    return _delta("la_delta_rule", q, k, v, beta, S0, y, S_out, None)


def delta_chunked_workspace_bytes(B, H, T) -> int:
    return int(_native.lib().la_delta_chunked_workspace_bytes(B, H, T))


def delta_rule_chunked(q, k, v, beta=None, S0=None, y=None, S_out=None, workspace=None):
    """The same memory in chunks of 64 tokens on the tensor cores (la_delta_rule_chunked):
    bf16 q, k [B,H,T,128], v [B,H,T,dv] with dv a multiple of 64; BF16 operands,
    FP32 state.  workspace: a device buffer of delta_chunked_workspace_bytes bytes
    (allocated here when None).  Returns (y [B,H,T,dv], S_T)."""
    B, H, T = q.shape[:3]
    if workspace is None and T > 0:
        workspace = torch.empty(delta_chunked_workspace_bytes(B, H, T), device=q.device, dtype=torch.uint8)
    return _delta("la_delta_rule_chunked", q, k, v, beta, S0, y, S_out, workspace)


def _delta(entry, q, k, v, beta, S0, y, S_out, workspace):
    if q.dtype not in _DTYPES:
        raise ValueError(f"unsupported dtype {q.dtype}")
    B, H, T, r = q.shape
    dv = v.shape[3]
    dev = q.device
    _require(q, "q", (B, H, T, r), q.dtype, dev)
    _require(k, "k", (B, H, T, r), q.dtype, dev)
    _require(v, "v", (B, H, T, dv), q.dtype, dev)
    _require(beta, "beta", (B, H, T), torch.float32, dev)
    _require(S0, "S0", (B, H, r, dv), torch.float32, dev)
    if y is None:
        y = torch.empty((B, H, T, dv), device=dev, dtype=q.dtype)
    if S_out is None:
        S_out = torch.empty((B, H, r, dv), device=dev, dtype=torch.float32)
    _require(y, "y", (B, H, T, dv), q.dtype, dev)
    _require(S_out, "S_out", (B, H, r, dv), torch.float32, dev)
    args = [_ptr(q), _ptr(k), _ptr(v), _DTYPES[q.dtype], _ptr(beta), _ptr(S0), B, H, T, r, dv, _ptr(y), _ptr(S_out)]
    if entry == "la_delta_rule_chunked":
        args += [_ptr(workspace), 0 if workspace is None else workspace.numel() * workspace.element_size()]
    with _device_guard(dev):
        st = getattr(_native.lib(), entry)(*args, _stream(dev))
    _native.check(st, entry)
    return y, S_out


def last_device_status(device="cuda") -> int:
    """Synchronises the current stream and returns (and clears) the device status word."""
    dev = torch.device(device)
    with _device_guard(dev):
        return int(_native.lib().la_last_device_status(_stream(dev)))
