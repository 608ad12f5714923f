"""ctypes wrapper around ``linattn_oracle.c`` (test infrastructure only).

The C file holds every step of the oracle's arithmetic; this module only builds
it with gcc, decodes argument types and allocates the FP64 result arrays.

Input arrays are numpy arrays in one of three element types, passed to C
without conversion:
  * float64, float32: used as is (widened to double inside C);
  * uint16: the raw bits of bfloat16 values (decoded exactly inside C).
Gates, initial states and results are float64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "linattn_oracle.c")
_LIB = os.path.join(_HERE, "liblinattn_oracle.so")

PHI_ELU1, PHI_RELU1, PHI_IDENTITY = 0, 1, 2
_IN_F64, _IN_F32, _IN_BF16 = 0, 1, 2

_lock = threading.Lock()
_default = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile the oracle with gcc (portable flags: no FMA contraction, no -march)."""
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
               "-shared", "-o", tmp, src, "-lpthread", "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)
    return out


def _bind(path: str):
    lib = ctypes.CDLL(path)
    vp, dp, i, d = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_double
    common = [i, i, i, i, i, vp, vp, vp, i, dp, dp, dp, d, i]
    lib.or_scan.argtypes = common + [i, dp, dp, dp]
    lib.or_dense.argtypes = common + [dp, dp, dp]
    lib.or_chunkwise.argtypes = common + [i, dp, dp, dp]
    lib.or_delta.argtypes = [i, i, i, i, i, vp, vp, vp, i, dp, dp, i, dp, dp]
    lib.or_backward.argtypes = common + [dp, dp, dp, i, dp, dp, dp, dp, dp, dp]
    for f in (lib.or_scan, lib.or_dense, lib.or_chunkwise, lib.or_delta, lib.or_backward):
        f.restype = ctypes.c_int
    lib.or_num_cpus.restype = ctypes.c_int
    return lib


def _load():
    global _default
    with _lock:
        if _default is None:
            _default = _bind(build())
    return _default


def variant(path: str) -> "Variant":
    """An oracle compiled from another source file (used by the tests that plant
    a mistake in a copy of the oracle and check that the pins catch it)."""
    return Variant(_bind(path))


def num_cpus() -> int:
    return int(_load().or_num_cpus())


def _in_type(a: np.ndarray) -> int:
    if a.dtype == np.float64:
        return _IN_F64
    if a.dtype == np.float32:
        return _IN_F32
    if a.dtype == np.uint16:
        return _IN_BF16
    raise TypeError(f"oracle input dtype {a.dtype} not supported")


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _prepare(q, k, v, alpha, S0, z0):
    q, k, v = (np.ascontiguousarray(x) for x in (q, k, v))
    if q.dtype != k.dtype or q.dtype != v.dtype:
        raise TypeError("q, k, v must share one dtype")
    if q.ndim != 4 or k.shape != q.shape or v.ndim != 4 or v.shape[:3] != q.shape[:3]:
        raise ValueError("expected q, k [B,H,T,r] and v [B,H,T,dv]")
    B, H, T, r = q.shape
    dv = v.shape[3]
    if alpha is not None:
        alpha = np.ascontiguousarray(alpha, dtype=np.float64).reshape(B, H, T)
    if S0 is not None:
        S0 = np.ascontiguousarray(S0, dtype=np.float64).reshape(B, H, r, dv)
    if z0 is not None:
        z0 = np.ascontiguousarray(z0, dtype=np.float64).reshape(B, H, r)
    return q, k, v, alpha, S0, z0, (B, H, T, r, dv)


def _outputs(B, H, T, r, dv):
    return (np.empty((B, H, T, dv)), np.empty((B, H, r, dv)), np.empty((B, H, r)))


def scan(q, k, v, alpha=None, S0=None, z0=None, eps=1e-6, phi=PHI_ELU1, threads=0, _lib=None):
    """Token recurrence; returns (y, S_T, z_T) in float64."""
    q, k, v, alpha, S0, z0, (B, H, T, r, dv) = _prepare(q, k, v, alpha, S0, z0)
    y, S, z = _outputs(B, H, T, r, dv)
    rc = (_lib or _load()).or_scan(B, H, T, r, dv, _ptr(q), _ptr(k), _ptr(v), _in_type(q), _ptr(alpha),
                         _ptr(S0), _ptr(z0), float(eps), int(phi), int(threads),
                         _ptr(y), _ptr(S), _ptr(z))
    if rc:
        raise ValueError("or_scan rejected its arguments")
    return y, S, z


def dense(q, k, v, alpha=None, S0=None, z0=None, eps=1e-6, phi=PHI_ELU1, _lib=None):
    """Quadratic masked form (tiny inputs only); returns (y, S_T, z_T)."""
    q, k, v, alpha, S0, z0, (B, H, T, r, dv) = _prepare(q, k, v, alpha, S0, z0)
    y, S, z = _outputs(B, H, T, r, dv)
    rc = (_lib or _load()).or_dense(B, H, T, r, dv, _ptr(q), _ptr(k), _ptr(v), _in_type(q), _ptr(alpha),
                          _ptr(S0), _ptr(z0), float(eps), int(phi), _ptr(y), _ptr(S), _ptr(z))
    if rc:
        raise ValueError("or_dense rejected its arguments")
    return y, S, z


def chunkwise(q, k, v, chunk, alpha=None, S0=None, z0=None, eps=1e-6, phi=PHI_ELU1, _lib=None):
    """Chunk formula with chunk size ``chunk``; returns (y, S_T, z_T)."""
    q, k, v, alpha, S0, z0, (B, H, T, r, dv) = _prepare(q, k, v, alpha, S0, z0)
    y, S, z = _outputs(B, H, T, r, dv)
    rc = (_lib or _load()).or_chunkwise(B, H, T, r, dv, _ptr(q), _ptr(k), _ptr(v), _in_type(q), _ptr(alpha),
                              _ptr(S0), _ptr(z0), float(eps), int(phi), int(chunk),
                              _ptr(y), _ptr(S), _ptr(z))
    if rc:
        raise ValueError("or_chunkwise rejected its arguments")
    return y, S, z


def backward(q, k, v, dy, alpha=None, S0=None, z0=None, dS_T=None, dz_T=None, eps=1e-6, phi=PHI_ELU1, threads=0,
             _lib=None):
    """Gradients of or_scan's outputs (y, S_T, z_T) for a loss with the given output
    gradients dy [B,H,T,dv] and, optionally, dS_T [B,H,r,dv], dz_T [B,H,r].
    Returns (dq, dk, dv, dalpha or None, dS0, dz0) in float64."""
    q, k, v, alpha, S0, z0, (B, H, T, r, dv) = _prepare(q, k, v, alpha, S0, z0)
    dy = np.ascontiguousarray(dy, dtype=np.float64).reshape(B, H, T, dv)
    if dS_T is not None:
        dS_T = np.ascontiguousarray(dS_T, dtype=np.float64).reshape(B, H, r, dv)
    if dz_T is not None:
        dz_T = np.ascontiguousarray(dz_T, dtype=np.float64).reshape(B, H, r)
    dq, dk = np.empty((B, H, T, r)), np.empty((B, H, T, r))
    dvo, dS0, dz0 = np.empty((B, H, T, dv)), np.empty((B, H, r, dv)), np.empty((B, H, r))
    dalpha = np.empty((B, H, T)) if alpha is not None else None
    rc = (_lib or _load()).or_backward(B, H, T, r, dv, _ptr(q), _ptr(k), _ptr(v), _in_type(q), _ptr(alpha),
                                       _ptr(S0), _ptr(z0), float(eps), int(phi), _ptr(dy), _ptr(dS_T),
                                       _ptr(dz_T), int(threads), _ptr(dq), _ptr(dk), _ptr(dvo), _ptr(dalpha),
                                       _ptr(dS0), _ptr(dz0))
    if rc:
        raise ValueError("or_backward rejected its arguments")
    return dq, dk, dvo, dalpha, dS0, dz0


def delta(q, k, v, beta=None, S0=None, threads=0, _lib=None):
    """Delta-rule memory (LA "Delta rule：先读旧答案，再写误差"): returns (y, S_T) in float64."""
    q, k, v, beta, S0, _, (B, H, T, r, dv) = _prepare(q, k, v, beta, S0, None)
    y, S = np.empty((B, H, T, dv)), np.empty((B, H, r, dv))
    rc = (_lib or _load()).or_delta(B, H, T, r, dv, _ptr(q), _ptr(k), _ptr(v), _in_type(q), _ptr(beta), _ptr(S0),
                                    int(threads), _ptr(y), _ptr(S))
    if rc:
        raise ValueError("or_delta rejected its arguments")
    return y, S


class Variant:
    """The three routes bound to one compiled copy of the oracle."""

    PHI_ELU1, PHI_RELU1, PHI_IDENTITY = PHI_ELU1, PHI_RELU1, PHI_IDENTITY

    def __init__(self, lib):
        self._lib = lib

    def scan(self, *a, **kw):
        return scan(*a, _lib=self._lib, **kw)

    def dense(self, *a, **kw):
        return dense(*a, _lib=self._lib, **kw)

    def chunkwise(self, *a, **kw):
        return chunkwise(*a, _lib=self._lib, **kw)

    def delta(self, *a, **kw):
        return delta(*a, _lib=self._lib, **kw)

    def backward(self, *a, **kw):
        return backward(*a, _lib=self._lib, **kw)
