"""Seeded synthetic inputs for the linear-attention path.

This module only draws random numbers and lays them out; it contains none of
the method's arithmetic.  Both the CUDA path (tests, benchmark) and the CPU
oracle (tests) are fed from it, so that both sides see identical bits.

Recipe: torch CPU generator seeded per workload; normal draws in FP32 (FP64
for the tiny FP64 workload), scaled, then rounded once to the workload dtype.
Gates are alpha = sigmoid(g), g ~ N(mu, sigma), computed in FP64 and rounded to
FP32; the gate is an input of the method, given per head and per token.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    T: int
    r: int = 128
    dv: int = 128
    dtype: torch.dtype = torch.bfloat16
    scale: float = 1.0          # standard deviation of q, k, v
    gated: bool = False         # alpha = sigmoid(N(gate_mu, gate_sigma)) per head and token
    gate_mu: float = 3.0
    gate_sigma: float = 1.0
    chunk: int = 64
    eps: float = 1e-6
    seed: int = 0
    decode: bool = False        # one token per request on a pre-existing state
    draw_fp64: bool = False     # draw in FP64 before rounding to ``dtype``
    lens: tuple = ()            # packed sequences: the length of each (B of them, T in total)

    @property
    def token_heads(self) -> int:
        return self.B * self.H * self.T

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The five workloads of the method's measurement plan, seeds 0..4 in this order.
TINY = Workload("tiny B1 H1 T64 r=dv=16 fp64->fp32", B=1, H=1, T=64, r=16, dv=16,
                dtype=torch.float32, draw_fp64=True, seed=0)
UNGATED = Workload("prefill B4 H16 T4096 d128 bf16 C64", B=4, H=16, T=4096, seed=1)
GATED = Workload("gated prefill B2 H16 T16384 d128 bf16 alpha=sigmoid(N(3,1))", B=2, H=16,
                 T=16384, gated=True, seed=2)
DECODE = Workload("decode B256 H16 r=dv=128 bf16 qkv, fp32 state", B=256, H=16, T=1,
                  decode=True, seed=3)
LONG = Workload("long prefill B1 H32 T65536 d128 bf16 sigma=2 C64", B=1, H=32, T=65536,
                scale=2.0, seed=4)
WORKLOADS = {"tiny": TINY, "ungated": UNGATED, "gated": GATED, "decode": DECODE, "long": LONG}

# The delta-rule memory on the shape of the ungated prefill.
DELTA = Workload("delta rule B4 H16 T4096 d128 bf16, unit q and k, beta=sigmoid(N(0,1))", B=4, H=16, T=4096,
                 seed=5)

# A short continuation: 8 tokens per request on a carried state (the decode
# requests' state distribution), gated; the state (256 MiB) exceeds L2.
def _loguniform_lens(n, lo, hi, seed):
    g = torch.Generator().manual_seed(seed)
    u = torch.rand(n, generator=g, dtype=torch.float64)
    return tuple(int(x) for x in torch.exp(u * (torch.log(torch.tensor(float(hi))) - torch.log(torch.tensor(float(lo))))
                                             + torch.log(torch.tensor(float(lo)))))


# Packed serving batches (la_prefill_varlen, token-major, from zero states, no gate):
# one long prompt among short ones, and prompt lengths spread log-uniformly.
_LONG_MIX = (16384,) + (512,) * 47
VARLEN_LONG = Workload("varlen one prompt of 16384 + 47 of 512 tokens H16 d128 bf16", B=len(_LONG_MIX), H=16,
                       T=sum(_LONG_MIX), lens=_LONG_MIX, seed=7)
_LOGU_MIX = _loguniform_lens(48, 128, 8192, seed=8)
_SHORT_MIX = tuple(int(x) for x in torch.randint(1, 33, (256,), generator=torch.Generator().manual_seed(9)))
VARLEN_LOGU = Workload("varlen 48 prompts of log-uniform 128..8192 tokens H16 d128 bf16", B=48, H=16,
                       T=sum(_LOGU_MIX), lens=_LOGU_MIX, seed=8)
# Ragged short continuations: 256 requests of 1..32 new tokens each (uniform,
# seeded), gated, each from its own carried state (the decode requests' state
# distribution), in place.
VARLEN_SHORT = Workload("varlen 256 short continuations of 1..32 tokens H16 d128 bf16 gated, fp32 states", B=256,
                        H=16, T=sum(_SHORT_MIX), lens=_SHORT_MIX, gated=True, decode=True, seed=9)

SHORT = Workload("short continuation B256 H16 T8 d128 bf16 alpha=sigmoid(N(3,1)), fp32 state", B=256, H=16, T=8,
                 gated=True, seed=6)


def prefill_inputs(w: Workload, device="cpu", with_state: bool = False, seed: int | None = None):
    """q, k [B,H,T,r], v [B,H,T,dv] in ``w.dtype``; alpha [B,H,T] FP32 or None;
    S0 [B,H,r,dv], z0 [B,H,r] FP32 (only when ``with_state``, else None).
    The carried-in state, when asked for, is the one of a decode request:
    S0 ~ N(0,1)*0.1 and z0 ~ U(1,100)."""
    g = torch.Generator().manual_seed(w.seed if seed is None else seed)
    draw_dtype = torch.float64 if w.draw_fp64 else torch.float32
    shape_qk = (w.B, w.H, w.T, w.r)
    shape_v = (w.B, w.H, w.T, w.dv)
    q = (torch.randn(shape_qk, generator=g, dtype=draw_dtype) * w.scale).to(w.dtype)
    k = (torch.randn(shape_qk, generator=g, dtype=draw_dtype) * w.scale).to(w.dtype)
    v = (torch.randn(shape_v, generator=g, dtype=draw_dtype) * w.scale).to(w.dtype)
    alpha = None
    if w.gated:
        gl = torch.randn((w.B, w.H, w.T), generator=g, dtype=torch.float64) * w.gate_sigma + w.gate_mu
        alpha = torch.sigmoid(gl).to(torch.float32)
    S0 = z0 = None
    if with_state:
        S0 = torch.randn((w.B, w.H, w.r, w.dv), generator=g, dtype=torch.float32) * 0.1
        z0 = torch.rand((w.B, w.H, w.r), generator=g, dtype=torch.float32) * 99.0 + 1.0
    out = dict(q=q, k=k, v=v, alpha=alpha, S0=S0, z0=z0)
    if device != "cpu":
        out = {n: (t.to(device) if t is not None else None) for n, t in out.items()}
    return out


def varlen_inputs(w: Workload, device="cpu", seed: int | None = None):
    """Packed sequences of lengths ``w.lens``: q, k [T, H, r], v [T, H, dv] in
    ``w.dtype`` (token-major, T = sum of the lengths), drawn as ``prefill_inputs``
    draws one sequence of T tokens; cu_seqlens int32 [B + 1]; with a gate, alpha
    [T, H] FP32; with ``w.decode`` (carried states), S0 [B,H,r,dv] ~ N(0,1)*0.1 and
    z0 [B,H,r] ~ U(1,100), FP32."""
    one = prefill_inputs(w.with_(B=1, T=sum(w.lens)), seed=seed)
    tok = lambda x: x[0].permute(1, 0, 2).contiguous()
    cu = torch.zeros(len(w.lens) + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(w.lens, dtype=torch.int64), 0).to(torch.int32)
    out = dict(q=tok(one["q"]), k=tok(one["k"]), v=tok(one["v"]), cu_seqlens=cu)
    if w.gated:
        out["alpha"] = one["alpha"][0].permute(1, 0).contiguous()
    if w.decode:
        g = torch.Generator().manual_seed((w.seed if seed is None else seed) + 1)
        B = len(w.lens)
        out["S0"] = torch.randn((B, w.H, w.r, w.dv), generator=g, dtype=torch.float32) * 0.1
        out["z0"] = torch.rand((B, w.H, w.r), generator=g, dtype=torch.float32) * 99.0 + 1.0
    if device != "cpu":
        out = {n: t.to(device) for n, t in out.items()}
    return out


def decode_inputs(w: Workload, device="cpu", seed: int | None = None):
    """One token per request: q, k [B,H,1,r], v [B,H,1,dv] in ``w.dtype``;
    pre-existing state S [B,H,r,dv] ~ N(0,1)*0.1 and z [B,H,r] ~ U(1,100), FP32;
    alpha [B,H] FP32 when gated, else None."""
    g = torch.Generator().manual_seed(w.seed if seed is None else seed)
    q = torch.randn((w.B, w.H, 1, w.r), generator=g, dtype=torch.float32).mul(w.scale).to(w.dtype)
    k = torch.randn((w.B, w.H, 1, w.r), generator=g, dtype=torch.float32).mul(w.scale).to(w.dtype)
    v = torch.randn((w.B, w.H, 1, w.dv), generator=g, dtype=torch.float32).mul(w.scale).to(w.dtype)
    S = torch.randn((w.B, w.H, w.r, w.dv), generator=g, dtype=torch.float32) * 0.1
    z = torch.rand((w.B, w.H, w.r), generator=g, dtype=torch.float32) * 99.0 + 1.0
    alpha = None
    if w.gated:
        gl = torch.randn((w.B, w.H), generator=g, dtype=torch.float64) * w.gate_sigma + w.gate_mu
        alpha = torch.sigmoid(gl).to(torch.float32)
    out = dict(q=q, k=k, v=v, alpha=alpha, S=S, z=z)
    if device != "cpu":
        out = {n: (t.to(device) if t is not None else None) for n, t in out.items()}
    return out


def delta_inputs(w: Workload, device="cpu", with_state: bool = False, seed: int | None = None):
    """Inputs of the delta-rule memory: q, k [B,H,T,r] drawn N(0,1) and divided by
    their Euclidean norm in FP32 (unit vectors, as in the pages' examples, so that
    beta |k|^2 = beta < 1 keeps every write a contraction), v [B,H,T,dv] ~
    N(0, scale^2), all rounded once to ``w.dtype``; beta [B,H,T] = sigmoid(N(0,1))
    in FP64 rounded to FP32; S0 [B,H,r,dv] ~ N(0,1)*0.1 when ``with_state``."""
    g = torch.Generator().manual_seed(w.seed if seed is None else seed)
    shape_qk = (w.B, w.H, w.T, w.r)
    unit = lambda x: x / x.norm(dim=-1, keepdim=True).clamp_min(1e-30)
    q = unit(torch.randn(shape_qk, generator=g, dtype=torch.float32)).to(w.dtype)
    k = unit(torch.randn(shape_qk, generator=g, dtype=torch.float32)).to(w.dtype)
    v = (torch.randn((w.B, w.H, w.T, w.dv), generator=g, dtype=torch.float32) * w.scale).to(w.dtype)
    beta = torch.sigmoid(torch.randn((w.B, w.H, w.T), generator=g, dtype=torch.float64)).to(torch.float32)
    S0 = torch.randn((w.B, w.H, w.r, w.dv), generator=g, dtype=torch.float32) * 0.1 if with_state else None
    out = dict(q=q, k=k, v=v, beta=beta, S0=S0)
    if device != "cpu":
        out = {n: (t.to(device) if t is not None else None) for n, t in out.items()}
    return out
