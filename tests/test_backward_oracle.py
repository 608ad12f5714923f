"""Pins of the FP64 backward oracle (oracle.backward) to facts fixed outside it.

The pages give no backward formula.  What fixes the gradients is the forward
itself: for L = sum(dy * y) + <dS_T, S_T> + <dz_T, z_T>, each gradient is the
derivative of L through the token recurrence (LA = "Linear attention：把历史写进状态",
sections "公式里的每个维度" and "加一个门：让旧记忆逐渐淡出").  The pins:
  - central finite differences of the forward oracle (or_scan), every input entry;
  - torch.autograd through an independent FP64 PyTorch loop written here;
  - exact special cases (a zero gate cuts S0, z0 off; zero output gradients).
Each check is a function of an oracle object so that planted mistakes in a
mutated copy of the C file are caught by the same checks."""
import os

import numpy as np
import pytest
import torch

import oracle as oracle_pkg

_ORACLE_SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "linattn_oracle.c")
EPS = 1e-6


def _problem(seed, B=1, H=2, T=7, r=3, dv=4, gated=True, zero_gate_at=None, state=True, scale=0.8):
    rng = np.random.default_rng(seed)
    d = dict(q=rng.standard_normal((B, H, T, r)) * scale, k=rng.standard_normal((B, H, T, r)) * scale,
             v=rng.standard_normal((B, H, T, dv)))
    d["alpha"] = rng.uniform(0.5, 1.0, (B, H, T)) if gated else None
    if zero_gate_at is not None:
        d["alpha"][:, :, zero_gate_at] = 0.0
    d["S0"] = rng.standard_normal((B, H, r, dv)) * 0.3 if state else None
    d["z0"] = rng.uniform(0.5, 2.0, (B, H, r)) if state else None
    d["dy"] = rng.standard_normal((B, H, T, dv))
    d["dS_T"] = rng.standard_normal((B, H, r, dv)) if state else None
    d["dz_T"] = rng.standard_normal((B, H, r)) if state else None
    return d


def _loss(o, d):
    y, S, z = o.scan(d["q"], d["k"], d["v"], alpha=d["alpha"], S0=d["S0"], z0=d["z0"], eps=EPS, threads=1)
    L = float(np.sum(d["dy"] * y))
    if d["dS_T"] is not None:
        L += float(np.sum(d["dS_T"] * S)) + float(np.sum(d["dz_T"] * z))
    return L


def _grads(o, d):
    dq, dk, dv, da, dS0, dz0 = o.backward(d["q"], d["k"], d["v"], d["dy"], alpha=d["alpha"], S0=d["S0"],
                                          z0=d["z0"], dS_T=d["dS_T"], dz_T=d["dz_T"], eps=EPS, threads=1)
    return dict(q=dq, k=dk, v=dv, alpha=da, S0=dS0, z0=dz0)


def check_finite_differences(o):
    """Every entry of every gradient against a central difference of the forward oracle."""
    for d in (_problem(1), _problem(2, zero_gate_at=3), _problem(3, gated=False, state=False, T=5)):
        g = _grads(o, d)
        for name in ("q", "k", "v", "alpha", "S0", "z0"):
            x = d[name]
            if x is None:
                assert g[name] is None or name in ("S0", "z0")
                continue
            num = np.empty_like(x)
            for idx in np.ndindex(x.shape):
                h = 1e-6 * max(1.0, abs(x[idx]))
                old = x[idx]
                x[idx] = old + h
                lp = _loss(oracle_pkg, d)
                x[idx] = old - h
                lm = _loss(oracle_pkg, d)
                x[idx] = old
                num[idx] = (lp - lm) / (2 * h)
            err = np.max(np.abs(num - g[name])) / max(1.0, np.max(np.abs(num)))
            assert err < 1e-6, (name, err)


def _torch_forward(q, k, v, alpha, S0, z0):
    """The recurrence written plainly in FP64 PyTorch (independent of the oracle)."""
    phi = lambda x: torch.where(x > 0, x + 1.0, torch.exp(torch.clamp(x, max=0.0)))
    B, H, T, r = q.shape
    S = S0.clone() if S0 is not None else torch.zeros(B, H, r, v.shape[-1], dtype=torch.float64)
    z = z0.clone() if z0 is not None else torch.zeros(B, H, r, dtype=torch.float64)
    ys = []
    for t in range(T):
        a = alpha[:, :, t, None] if alpha is not None else 1.0
        kt, qt = phi(k[:, :, t]), phi(q[:, :, t])
        S = (a[..., None] if alpha is not None else 1.0) * S + kt[..., :, None] * v[:, :, t, None, :]
        z = a * z + kt
        ys.append(torch.einsum("bhi,bhij->bhj", qt, S) / (torch.einsum("bhi,bhi->bh", qt, z) + EPS)[..., None])
    return torch.stack(ys, dim=2), S, z


def check_autograd(o):
    d = _problem(4, B=2, H=1, T=9, r=4, dv=3)
    g = _grads(o, d)
    names = ("q", "k", "v", "alpha", "S0", "z0")
    ts = {n: torch.tensor(d[n], requires_grad=True) for n in names}
    y, S, z = _torch_forward(*(ts[n] for n in names))
    L = (torch.tensor(d["dy"]) * y).sum() + (torch.tensor(d["dS_T"]) * S).sum() + (torch.tensor(d["dz_T"]) * z).sum()
    auto = torch.autograd.grad(L, [ts[n] for n in names])
    for n, a in zip(names, auto):
        assert np.allclose(g[n], a.numpy(), rtol=1e-10, atol=1e-12), n


def check_special_cases(o):
    # a zero gate on the first token: nothing flows back into S0, z0
    d = _problem(5, zero_gate_at=0)
    g = _grads(o, d)
    assert not g["S0"].any() and not g["z0"].any()
    # no output gradient: every gradient is zero
    d = _problem(6)
    d["dy"][:] = 0.0
    d["dS_T"][:] = 0.0
    d["dz_T"][:] = 0.0
    g = _grads(o, d)
    assert all(not g[n].any() for n in ("q", "k", "v", "alpha", "S0", "z0"))
    # only dS_T: with no output read, dS0 = (product of all gates) dS_T
    d = _problem(7)
    d["dy"][:] = 0.0
    d["dz_T"][:] = 0.0
    g = _grads(o, d)
    prod = np.prod(d["alpha"], axis=2)[..., None, None]
    assert np.allclose(g["S0"], prod * d["dS_T"], rtol=1e-13)


ALL_CHECKS = [(f.__name__, f) for f in (check_finite_differences, check_autograd, check_special_cases)]


@pytest.mark.parametrize("name,check", ALL_CHECKS, ids=[n for n, _ in ALL_CHECKS])
def test_backward_pins(name, check):
    check(oracle_pkg)


def test_backward_long_sequence_segments():
    """T spanning several recomputation segments gives the same gradients as a
    short-segment-free reference (the autograd loop) on a longer sequence."""
    d = _problem(8, B=1, H=1, T=150, r=3, dv=2)
    g = _grads(oracle_pkg, d)
    names = ("q", "k", "v", "alpha", "S0", "z0")
    ts = {n: torch.tensor(d[n], requires_grad=True) for n in names}
    y, S, z = _torch_forward(*(ts[n] for n in names))
    L = (torch.tensor(d["dy"]) * y).sum() + (torch.tensor(d["dS_T"]) * S).sum() + (torch.tensor(d["dz_T"]) * z).sum()
    for n, a in zip(names, torch.autograd.grad(L, [ts[n] for n in names])):
        assert np.allclose(g[n], a.numpy(), rtol=1e-9, atol=1e-12), n


MUTATIONS = [
    ("dd term dropped", "double aq = dd * zt[i], ak = g[i];", "double aq = 0.0 * zt[i], ak = g[i];"),
    ("gate applied before the read", "            for (size_t x = 0; x < rd; ++x) G[x] *= a;\n",
     "            for (size_t x = 0; x < rd; ++x) G[x] *= a * a;\n"),
    ("dalpha from S_t", "for (size_t x = 0; x < rd; ++x) da += G[x] * Sp[x];", "for (size_t x = 0; x < rd; ++x) da += G[x] * St[x];"),
    ("phi' of ELU", "if (kind == OR_PHI_ELU1) return x > 0.0 ? 1.0 : exp(x);", "if (kind == OR_PHI_ELU1) return 1.0;"),
    ("denominator sign", "dd -= bp->dy[row_v + j] * w->y[(size_t)t * dv + j];", "dd += bp->dy[row_v + j] * w->y[(size_t)t * dv + j];"),
    ("z gradient of k dropped", "double aq = dd * zt[i], ak = g[i];", "double aq = dd * zt[i], ak = 0.0;"),
]


@pytest.mark.parametrize("desc,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_backward_mistakes_are_caught(tmp_path, desc, old, new):
    src = open(_ORACLE_SRC).read()
    assert old in src, f"mutation anchor missing: {old}"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    mutant = oracle_pkg.variant(oracle_pkg.build(force=True, src=str(path), out=str(tmp_path / "libmutant.so")))
    caught = []
    for name, check in ALL_CHECKS:
        try:
            check(mutant)
        except (AssertionError, ValueError, FloatingPointError):
            caught.append(name)
    assert caught, f"no pin catches the planted mistake: {desc}"
