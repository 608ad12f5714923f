"""Backward pass on the GPU (la_prefill_backward) against the FP64 oracle's gradients
(oracle.backward, pinned by finite differences in test_backward_oracle.py).

The backward takes the forward's output y.  In test_backward_parity y comes from
the oracle, rounded to the I/O type, so that those cases do not depend on the
forward kernels; test_backward_after_gpu_forward and the full-size case run the
GPU forward into the GPU backward, as training does.
Tolerances (max |gpu - ref| / max |ref| per tensor): BF16 inputs 2e-2 (dq, dk,
dv are rounded to BF16, and dd_t uses the BF16 y); FP32 inputs 1e-4 (FP32
accumulation over T tokens in three sweeps, and dalpha is formed as a
difference of running sums divided by alpha)."""
import numpy as np
import pytest
import torch

from conftest import assert_close, max_rel_err, row_rel_err, to_oracle

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}
EPS = 1e-6


@pytest.fixture(scope="module")
def la():
    from recurrent_state_02_gb300 import build
    build.build()
    import recurrent_state_02_gb300 as la_mod
    assert torch.cuda.is_available()
    return la_mod


def _case(oracle_mod, B, H, T, r, dv, dtype, gated, with_state, seed):
    from recurrent_state_02_gb300 import workloads as W
    w = W.Workload("bwd", B=B, H=H, T=T, r=r, dv=dv, dtype=dtype, gated=gated, seed=seed)
    d = W.prefill_inputs(w, with_state=with_state)
    g = torch.Generator().manual_seed(seed + 1)
    d["dy"] = torch.randn((B, H, T, dv), generator=g).to(dtype)
    d["dS_T"] = torch.randn((B, H, r, dv), generator=g) * 0.1 if with_state else None
    d["dz_T"] = torch.randn((B, H, r), generator=g) * 0.1 if with_state else None
    args = [to_oracle(d[n]) for n in ("q", "k", "v")]
    y, _, _ = oracle_mod.scan(*args, alpha=to_oracle(d["alpha"]), S0=to_oracle(d["S0"]), z0=to_oracle(d["z0"]),
                              eps=EPS, threads=0)
    d["y"] = torch.from_numpy(y).to(dtype)
    ref = oracle_mod.backward(*args, d["dy"].double().numpy(), alpha=to_oracle(d["alpha"]), S0=to_oracle(d["S0"]),
                              z0=to_oracle(d["z0"]), dS_T=to_oracle(d["dS_T"]), dz_T=to_oracle(d["dz_T"]), eps=EPS,
                              threads=0)
    return d, ref


def _gpu(la, d):
    g = {k: (v.cuda() if v is not None else None) for k, v in d.items()}
    out = la.prefill_backward(g["q"], g["k"], g["v"], g["y"], g["dy"], alpha=g["alpha"], S0=g["S0"], z0=g["z0"],
                              dS_T=g["dS_T"], dz_T=g["dz_T"], eps=EPS)
    assert la.last_device_status() == 0
    return [None if t is None else t.float().cpu().numpy() for t in out]


CASES = [
    # dtype, r, dv, T, gated, with_state
    (torch.float32, 128, 128, 200, True, True),
    (torch.float32, 64, 32, 75, False, True),
    (torch.float32, 32, 64, 33, True, False),
    (torch.float32, 128, 64, 1, True, True),
    (torch.bfloat16, 128, 128, 300, True, True),
    (torch.bfloat16, 128, 128, 97, False, False),
    (torch.bfloat16, 64, 128, 64, True, True),
]


@pytest.mark.parametrize("dtype,r,dv,T,gated,with_state", CASES,
                         ids=[f"{str(c[0])[6:]}-r{c[1]}-dv{c[2]}-T{c[3]}-g{int(c[4])}-S{int(c[5])}" for c in CASES])
def test_backward_parity(la, oracle_mod, dtype, r, dv, T, gated, with_state):
    d, ref = _case(oracle_mod, 2, 2, T, r, dv, dtype, gated, with_state, seed=300 + r + dv + T)
    got = _gpu(la, d)
    names = ("dq", "dk", "dv", "dalpha", "dS0", "dz0")
    for name, a, b in zip(names, got, ref):
        if b is None:
            assert a is None
            continue
        assert np.isfinite(a).all(), name
        err = max_rel_err(a, b)
        # per-row error reported only: a gradient row can be a near-cancelling
        # difference (dq_t ~ S_t dn_t - z_t (dy_t . y_t) / d_t), so its own size is
        # not the scale of its rounding
        print(f"[parity] backward {name}: tensor {err:.3e} row {row_rel_err(a, b):.3e}")
        assert err <= TOL[dtype], (name, err)


# BF16 at r = dv = 128 runs the three sweeps on the tensor cores: ragged lengths
# (T = 1, one chunk exactly, one token past it), zero gates at and around chunk
# boundaries, and gates that decay by more than e^-44 inside a chunk.
TC_EDGE = [
    # T, gated, with_state, gate edits
    (1, True, True, None),
    (64, False, True, None),
    (65, True, False, None),
    (200, True, True, "zeros"),
    (190, True, False, "tiny"),
]


@pytest.mark.parametrize("T,gated,with_state,edit", TC_EDGE,
                         ids=[f"T{c[0]}-g{int(c[1])}-S{int(c[2])}-{c[3]}" for c in TC_EDGE])
def test_backward_tc_edges(la, oracle_mod, T, gated, with_state, edit):
    from recurrent_state_02_gb300 import workloads as W
    B, H = 1, 3
    w = W.Workload("bwd-tc", B=B, H=H, T=T, dtype=torch.bfloat16, gated=gated, seed=500 + T)
    d = W.prefill_inputs(w, with_state=with_state)
    if edit == "zeros":
        for t in (0, 63, 64, 127, 150):
            d["alpha"][0, 0, t] = 0.0
        d["alpha"][0, 1, 70:90] = 0.0
    elif edit == "tiny":
        d["alpha"][0, 0, 64:128] = 0.2
        d["alpha"][0, 2, 100] = 1e-20
    g = torch.Generator().manual_seed(501 + T)
    dy = torch.randn((B, H, T, 128), generator=g).to(torch.bfloat16)
    dS_T = torch.randn((B, H, 128, 128), generator=g) * 0.1 if with_state else None
    dz_T = torch.randn((B, H, 128), generator=g) * 0.1 if with_state else None
    args = [to_oracle(d[n]) for n in ("q", "k", "v")]
    y, _, _ = oracle_mod.scan(*args, alpha=to_oracle(d["alpha"]), S0=to_oracle(d["S0"]), z0=to_oracle(d["z0"]),
                              eps=EPS)
    ref = oracle_mod.backward(*args, dy.double().numpy(), alpha=to_oracle(d["alpha"]), S0=to_oracle(d["S0"]),
                              z0=to_oracle(d["z0"]), dS_T=to_oracle(dS_T), dz_T=to_oracle(dz_T), eps=EPS, threads=0)
    gd = {k: (v.cuda() if v is not None else None) for k, v in d.items()}
    out = la.prefill_backward(gd["q"], gd["k"], gd["v"], torch.from_numpy(y).to(torch.bfloat16).cuda(), dy.cuda(),
                              alpha=gd["alpha"], S0=gd["S0"], z0=gd["z0"],
                              dS_T=dS_T.cuda() if dS_T is not None else None,
                              dz_T=dz_T.cuda() if dz_T is not None else None, eps=EPS)
    assert la.last_device_status() == 0
    for name, a, r_ in zip(("dq", "dk", "dv", "dalpha", "dS0", "dz0"), out, ref):
        if r_ is None:
            assert a is None
            continue
        a = a.float().cpu().numpy()
        if name == "dalpha":
            # dalpha_u is the log-gate derivative over alpha_u: defined where alpha_u > 0,
            # and its absolute error grows as 1 / alpha_u, so the bar covers alpha_u >= 0.05
            keep = d["alpha"].numpy() >= 0.05
            a, r_ = a[keep], r_[keep]
        assert np.isfinite(a).all(), name
        err = max_rel_err(a, r_)
        print(f"[parity] backward (tensor cores) {name}: tensor {err:.3e}")
        assert err <= 2e-2, (name, err)


# Long sequences over few heads run the tensor-core sweeps over sequence segments
# (at least 16 chunks each, as many as the SMs allow per head): the states
# entering each segment come from a forward state pass (dq) and a reversed one
# (dk, dv), whose parts the scans compose.  B*H = 2 or 3 on a GB300's 152 SMs
# gives 2 to 4 segments, and state-pass parts of a single chunk.
SEG_CASES = [
    # B, H, T, gated, with_state, gate edits
    (1, 2, 4100, True, True, None),
    (1, 3, 2113, False, False, None),
    (1, 2, 3200, True, False, "edges"),
]


@pytest.mark.parametrize("B,H,T,gated,with_state,edit", SEG_CASES,
                         ids=[f"B{c[0]}H{c[1]}T{c[2]}-g{int(c[3])}-S{int(c[4])}-{c[5]}" for c in SEG_CASES])
def test_backward_segmented(la, oracle_mod, B, H, T, gated, with_state, edit):
    from recurrent_state_02_gb300 import workloads as W
    w = W.Workload("bwd-seg", B=B, H=H, T=T, dtype=torch.bfloat16, gated=gated, seed=600 + T)
    d = W.prefill_inputs(w, with_state=with_state)
    if edit == "edges":
        # zero gates on the tokens either side of chunk and segment boundaries, and
        # a run of small gates across one
        for t in (0, 1023, 1024, 1087, 1088, 2175, 2176, T - 1):
            d["alpha"][0, 0, t] = 0.0
        d["alpha"][0, 1, 1000:1200] = 0.3
    g = torch.Generator().manual_seed(601 + T)
    dy = torch.randn((B, H, T, 128), generator=g).to(torch.bfloat16)
    dS_T = torch.randn((B, H, 128, 128), generator=g) * 0.1 if with_state else None
    dz_T = torch.randn((B, H, 128), generator=g) * 0.1 if with_state else None
    gd = {k: (v.cuda() if v is not None else None) for k, v in d.items()}
    # the GPU forward's y, as training feeds it
    y, _, _ = la.prefill_chunked(gd["q"], gd["k"], gd["v"], alpha=gd["alpha"], S0=gd["S0"], z0=gd["z0"], eps=EPS)
    args = [to_oracle(d[n]) for n in ("q", "k", "v")]
    ref = oracle_mod.backward(*args, dy.double().numpy(), alpha=to_oracle(d["alpha"]), S0=to_oracle(d["S0"]),
                              z0=to_oracle(d["z0"]), dS_T=to_oracle(dS_T), dz_T=to_oracle(dz_T), eps=EPS, threads=0)
    out = la.prefill_backward(gd["q"], gd["k"], gd["v"], y, dy.cuda(), alpha=gd["alpha"], S0=gd["S0"], z0=gd["z0"],
                              dS_T=dS_T.cuda() if dS_T is not None else None,
                              dz_T=dz_T.cuda() if dz_T is not None else None, eps=EPS)
    assert la.last_device_status() == 0
    for name, a, r_ in zip(("dq", "dk", "dv", "dalpha", "dS0", "dz0"), out, ref):
        if r_ is None:
            assert a is None
            continue
        a = a.float().cpu().numpy()
        if name == "dalpha":
            keep = d["alpha"].numpy() >= 0.05   # defined where alpha > 0; error grows as 1 / alpha
            a, r_ = a[keep], r_[keep]
        assert np.isfinite(a).all(), name
        err = max_rel_err(a, r_)
        print(f"[parity] segmented backward {name}: tensor {err:.3e}")
        assert err <= 2e-2, (name, err)


CHAIN_CASES = [
    # T, gated, with_state
    (300, True, True),
    (64 * 5 + 7, False, False),
]


@pytest.mark.parametrize("T,gated,with_state", CHAIN_CASES,
                         ids=[f"T{c[0]}-g{int(c[1])}-S{int(c[2])}" for c in CHAIN_CASES])
def test_backward_after_gpu_forward(la, oracle_mod, T, gated, with_state):
    """The training chain: y from the GPU forward (BF16 tensor-core prefill) feeds
    the GPU backward; the gradients are held to the oracle's, which recomputes y
    in FP64 itself."""
    from recurrent_state_02_gb300 import workloads as W
    B, H = 2, 3
    w = W.Workload("bwd-chain", B=B, H=H, T=T, dtype=torch.bfloat16, gated=gated, seed=400 + T)
    d = W.prefill_inputs(w, with_state=with_state)
    g = torch.Generator().manual_seed(401 + T)
    dy = torch.randn((B, H, T, 128), generator=g).to(torch.bfloat16)
    args = [to_oracle(d[n]) for n in ("q", "k", "v")]
    ref = oracle_mod.backward(*args, dy.double().numpy(), alpha=to_oracle(d["alpha"]), S0=to_oracle(d["S0"]),
                              z0=to_oracle(d["z0"]), eps=EPS, threads=0)
    gd = {k: (v.cuda() if v is not None else None) for k, v in d.items()}
    y, _, _ = la.prefill_chunked(gd["q"], gd["k"], gd["v"], alpha=gd["alpha"], S0=gd["S0"], z0=gd["z0"], eps=EPS)
    out = la.prefill_backward(gd["q"], gd["k"], gd["v"], y, dy.cuda(), alpha=gd["alpha"], S0=gd["S0"], z0=gd["z0"],
                              eps=EPS)
    assert la.last_device_status() == 0
    for name, a, r_ in zip(("dq", "dk", "dv", "dalpha", "dS0", "dz0"), out, ref):
        if r_ is None:
            assert a is None
            continue
        a = a.float().cpu().numpy()
        assert np.isfinite(a).all(), name
        err = max_rel_err(a, r_)
        print(f"[parity] forward->backward {name}: tensor {err:.3e} row {row_rel_err(a, r_):.3e}")
        assert err <= 2e-2, (name, err)


def test_backward_full_size_sampled_heads(la, oracle_mod):
    """B4 H16 T4096 r = dv = 128 BF16 with a gate, the shape the benchmark times;
    the oracle recomputes two sampled heads (heads are independent)."""
    from recurrent_state_02_gb300 import workloads as W
    w = W.UNGATED.with_(gated=True)
    d = W.prefill_inputs(w)
    g = torch.Generator().manual_seed(99)
    d["dy"] = torch.randn(d["v"].shape, generator=g).to(torch.bfloat16)
    heads = ((0, 0), (3, 11))
    refs = {}
    for b, h in heads:
        one = {n: (t[b:b + 1, h:h + 1].contiguous() if t is not None else None) for n, t in d.items()}
        args = [to_oracle(one[n]) for n in ("q", "k", "v")]
        y, _, _ = oracle_mod.scan(*args, alpha=to_oracle(one["alpha"]), eps=EPS)
        refs[(b, h)] = (y, oracle_mod.backward(*args, one["dy"].double().numpy(), alpha=to_oracle(one["alpha"]),
                                               eps=EPS))
    # y for every head from the GPU forward (the sampled heads are checked against the oracle's y too)
    gd = {k: (v.cuda() if v is not None else None) for k, v in d.items()}
    y, _, _ = la.prefill_chunked(gd["q"], gd["k"], gd["v"], alpha=gd["alpha"], eps=EPS)
    out = la.prefill_backward(gd["q"], gd["k"], gd["v"], y, gd["dy"], alpha=gd["alpha"], eps=EPS)
    assert la.last_device_status() == 0
    got = [t.float().cpu().numpy() for t in out]
    for (b, h), (y_ref, ref) in refs.items():
        assert_close(y[b:b + 1, h:h + 1].float().cpu().numpy(), y_ref, 2e-2, f"forward y head {b},{h}")
        for name, a, r_ in zip(("dq", "dk", "dv", "dalpha", "dS0", "dz0"), got, ref):
            err = max_rel_err(a[b:b + 1, h:h + 1], r_)
            assert err <= 2e-2, (name, b, h, err)


def test_backward_workspace_errors(la):
    q = torch.zeros(1, 1, 8, 32, device="cuda")
    v = torch.zeros(1, 1, 8, 32, device="cuda")
    small = torch.empty(16, device="cuda", dtype=torch.uint8)
    with pytest.raises(la.LinAttnError):
        la.prefill_backward(q, q, v, v, v, workspace=small)
