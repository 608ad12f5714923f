"""The saved denominator: la_prefill_chunked_save writes d_t = phi(q_t) . z_t + eps
(the normaliser of "公式里的每个维度", y_t = phi(q_t)^T S_t / d_t), and
la_prefill_backward_saved takes it instead of recomputing it.

- The gradients of the chain prefill_chunked_save -> prefill_backward(d=...) are
  held to the FP64 oracle's (oracle.backward, pinned by finite differences in
  test_backward_oracle.py), at the bars of test_gpu_backward.py.
- The forward's outputs are those of prefill_chunked, bit for bit.
- d itself is checked against its definition: z_t = alpha_t z_{t-1} + phi(k_t),
  written out below in FP64 on the inputs the kernels read.  BF16 bar 1e-2
  elementwise relative (d is a sum of positive terms; the chunk kernel forms it
  from BF16 operands, with phi in BF16), FP32 bar 1e-5.
- Where the backward splits the sequence into segments, the states the forward
  keeps for it are the oracle's states at chunk boundaries (its scan over the
  prefix), in increasing order, the first one S0, z0; bar 2e-2 of each state's
  largest entry.
"""
import numpy as np
import pytest
import torch

from conftest import max_rel_err, row_rel_err, to_oracle

pytestmark = pytest.mark.gpu

EPS = 1e-6
TOL_GRAD = {torch.float32: 1e-4, torch.bfloat16: 2e-2}
TOL_D = {torch.float32: 1e-5, torch.bfloat16: 1e-2}

CASES = [
    # dtype, B, H, T, r, dv, gated, with_state
    (torch.bfloat16, 2, 3, 300, 128, 128, True, True),
    (torch.bfloat16, 1, 2, 1000, 128, 64, False, False),
    (torch.bfloat16, 1, 2, 2500, 128, 128, True, False),   # few long sequences: sequence segments
    (torch.bfloat16, 1, 1, 65, 128, 128, True, True),      # ragged tail of one token
    (torch.bfloat16, 2, 2, 700, 128, 64, True, True),      # gated 64-column slices
    (torch.bfloat16, 2, 3, 9, 128, 128, True, True),       # a short continuation (the token walk)
    (torch.bfloat16, 2, 2, 25, 128, 128, True, True),      # the walk over two halves of 16 tokens
    (torch.bfloat16, 1, 2, 3000, 128, 128, False, True),   # ungated whole heads, segments, kept states
    (torch.float32, 2, 2, 200, 64, 64, True, True),
]


@pytest.fixture(scope="module")
def la():
    from recurrent_state_02_gb300 import build
    build.build()
    import recurrent_state_02_gb300 as la_mod
    assert torch.cuda.is_available()
    return la_mod


def _inputs(dtype, B, H, T, r, dv, gated, with_state, seed):
    from recurrent_state_02_gb300 import workloads as W
    w = W.Workload("saved-d", B=B, H=H, T=T, r=r, dv=dv, dtype=dtype, gated=gated, seed=seed)
    d = W.prefill_inputs(w, with_state=with_state)
    g = torch.Generator().manual_seed(seed + 1)
    d["dy"] = torch.randn((B, H, T, dv), generator=g).to(dtype)
    return d


def _d_by_definition(d):
    """d_t = phi(q_t) . z_t + eps, z_t = alpha_t z_{t-1} + phi(k_t), in FP64."""
    q, k = d["q"].double().numpy(), d["k"].double().numpy()
    phi = lambda x: np.where(x > 0, x + 1.0, np.exp(np.minimum(x, 0.0)))
    pq, pk = phi(q), phi(k)
    B, H, T, r = q.shape
    alpha = d["alpha"].double().numpy() if d["alpha"] is not None else np.ones((B, H, T))
    z = d["z0"].double().numpy().copy() if d["z0"] is not None else np.zeros((B, H, r))
    out = np.empty((B, H, T))
    for t in range(T):
        z = alpha[:, :, t, None] * z + pk[:, :, t]
        out[:, :, t] = np.einsum("bhi,bhi->bh", pq[:, :, t], z) + EPS
    return out


@pytest.mark.parametrize("dtype,B,H,T,r,dv,gated,with_state", CASES,
                         ids=[f"{str(c[0]).split('.')[-1]}-B{c[1]}H{c[2]}T{c[3]}-dv{c[5]}-g{int(c[6])}-s{int(c[7])}"
                              for c in CASES])
def test_saved_denominator_chain(la, oracle_mod, dtype, B, H, T, r, dv, gated, with_state):
    d = _inputs(dtype, B, H, T, r, dv, gated, with_state, seed=500 + T + dv)
    g = {n: (t.cuda() if t is not None else None) for n, t in d.items()}
    kw = dict(alpha=g["alpha"], S0=g["S0"], z0=g["z0"], eps=EPS)
    y, S_T, z_T, dn, states = la.prefill_chunked_save(g["q"], g["k"], g["v"], **kw)
    y0, S0_, z0_ = la.prefill_chunked(g["q"], g["k"], g["v"], **kw)
    assert la.last_device_status() == 0
    assert torch.equal(y, y0) and torch.equal(S_T, S0_) and torch.equal(z_T, z0_)

    ref_d = _d_by_definition(d)
    got_d = dn.cpu().double().numpy()
    assert np.isfinite(got_d).all() and (got_d > 0).all()
    d_err = float(np.max(np.abs(got_d - ref_d) / ref_d))
    print(f"[parity] saved d: elementwise relative {d_err:.3e}")
    assert d_err <= TOL_D[dtype], d_err

    if states is not None:
        _check_states(oracle_mod, d, states.cpu().double().numpy())
    out_saved = la.prefill_backward(g["q"], g["k"], g["v"], y, g["dy"], d=dn, states=states, **kw)
    out_plain = la.prefill_backward(g["q"], g["k"], g["v"], y, g["dy"], **kw)
    assert la.last_device_status() == 0
    args = [to_oracle(d[n]) for n in ("q", "k", "v")]
    ref = oracle_mod.backward(*args, d["dy"].double().numpy(), alpha=to_oracle(d["alpha"]), S0=to_oracle(d["S0"]),
                              z0=to_oracle(d["z0"]), eps=EPS, threads=0)
    for name, a, b, r_ in zip(("dq", "dk", "dv", "dalpha", "dS0", "dz0"), out_saved, out_plain, ref):
        if r_ is None:
            assert a is None and b is None
            continue
        a = a.float().cpu().numpy()
        b = b.float().cpu().numpy()
        assert np.isfinite(a).all(), name
        err = max_rel_err(a, r_)
        print(f"[parity] saved-d backward {name}: tensor {err:.3e} row {row_rel_err(a, r_):.3e}; "
              f"against the recomputing backward {max_rel_err(a, b):.3e}")
        assert err <= TOL_GRAD[dtype], (name, err)
        assert max_rel_err(a, b) <= TOL_GRAD[dtype], name


def _check_states(oracle_mod, d, flat):
    B, H, T, r = d["q"].shape
    dv = d["v"].shape[3]
    per = B * H * (r * dv + r)
    assert flat.size % per == 0
    nseg = flat.size // per
    assert nseg >= 2
    st = flat.reshape(nseg, B, H, r * dv + r)
    S = st[..., :r * dv].reshape(nseg, B, H, r, dv)
    z = st[..., r * dv:]
    S0 = d["S0"].double().numpy() if d["S0"] is not None else np.zeros((B, H, r, dv))
    z0 = d["z0"].double().numpy() if d["z0"] is not None else np.zeros((B, H, r))
    assert np.array_equal(S[0], S0) and np.array_equal(z[0], z0)
    # the oracle's state after every chunk boundary t0 (its scan over tokens [0, t0))
    cut = lambda t, t0: to_oracle(t[:, :, :t0].contiguous()) if t is not None else None
    prefix = {}
    for t0 in range(64, T, 64):
        _, Sr, zr = oracle_mod.scan(cut(d["q"], t0), cut(d["k"], t0), cut(d["v"], t0), alpha=cut(d["alpha"], t0),
                                    S0=to_oracle(d["S0"]), z0=to_oracle(d["z0"]), eps=EPS, threads=0)
        prefix[t0] = (Sr, zr)
    last = 0
    for gseg in range(1, nseg):
        errs = {t0: max(max_rel_err(S[gseg], Sr), max_rel_err(z[gseg], zr)) for t0, (Sr, zr) in prefix.items()}
        t0 = min(errs, key=errs.get)
        print(f"[parity] kept state {gseg}: token {t0}, relative {errs[t0]:.3e}")
        assert errs[t0] <= 2e-2 and t0 > last, (gseg, t0, errs[t0])
        last = t0
