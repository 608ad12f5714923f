"""Delta-rule memory on the GPU (la_delta_rule) against the FP64 oracle (oracle.delta).

LA = "Linear attention：把历史写进状态", section "Delta rule：先读旧答案，再写误差":
p = S^T k, S <- S + beta k (v - p)^T, y = S^T q after the write.  Inputs are the
seeded unit-key recipe of workloads.delta_inputs; both sides see the same bits.

Tolerances: the kernel computes in FP32 from the exact input values, so S_T
(FP32) is held to 1e-5 for both input types; y is held to 1e-5 on FP32 inputs
and to 2e-2 on BF16 inputs, where it is rounded to BF16 on output."""
import json
import os

import numpy as np
import pytest
import torch

from conftest import assert_close, to_oracle

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "delta_examples.json")
TOL_F32, TOL_BF16 = 1e-5, 2e-2


@pytest.fixture(scope="module")
def la():
    from recurrent_state_02_gb300 import build
    build.build()
    import recurrent_state_02_gb300 as la_mod
    assert torch.cuda.is_available()
    return la_mod


def _inputs(B, H, T, r, dv, dtype, with_state, with_beta, seed):
    from recurrent_state_02_gb300 import workloads as W
    w = W.Workload("delta-test", B=B, H=H, T=T, r=r, dv=dv, dtype=dtype, seed=seed)
    d = W.delta_inputs(w, with_state=with_state)
    if not with_beta:
        d["beta"] = None
    return d


def _oracle(oracle_mod, d):
    return oracle_mod.delta(to_oracle(d["q"]), to_oracle(d["k"]), to_oracle(d["v"]), beta=to_oracle(d["beta"]),
                            S0=to_oracle(d["S0"]), threads=0)


def _run(la, d):
    g = {k: (v.cuda() if v is not None else None) for k, v in d.items()}
    y, S = la.delta_rule(g["q"], g["k"], g["v"], beta=g["beta"], S0=g["S0"])
    assert la.last_device_status() == 0
    return y.float().cpu().numpy(), S.cpu().numpy()


def test_delta_pages_examples(la):
    """The pages' worked numbers, embedded in r = dv = 32 with zero padding (FP32,
    exact): orthogonal keys (the written key reads 3.5, the other keeps 4) and
    three writes of one key (3.5, 4.25, 4.625)."""
    cases = {c["name"]: c for c in json.load(open(GOLDEN))["cases"]}
    c = cases["orthogonal_keys"]
    r = dv = 32
    q = torch.zeros(2, 1, 1, r)
    q[0, 0, 0, 0] = 1.0   # request 0 queries the written key
    q[1, 0, 0, 1] = 1.0   # request 1 queries the orthogonal key
    k = torch.zeros(2, 1, 1, r)
    k[:, 0, 0, :2] = torch.tensor(c["k"][0], dtype=torch.float32)
    v = torch.zeros(2, 1, 1, dv)
    v[:, 0, 0, 0] = c["v"][0][0]
    S0 = torch.zeros(2, 1, r, dv)
    S0[:, 0, 0, 0], S0[:, 0, 1, 0] = c["S0"][0][0], c["S0"][1][0]
    beta = torch.full((2, 1, 1), c["beta"][0])
    y, S = _run(la, dict(q=q, k=k, v=v, beta=beta, S0=S0))
    assert y[0, 0, 0, 0] == c["S_final"][0][0] and y[1, 0, 0, 0] == c["S_final"][1][0]
    assert S[0, 0, 0, 0] == c["S_final"][0][0] and S[0, 0, 1, 0] == c["S_final"][1][0]
    assert np.count_nonzero(S[0, 0]) == 2 and np.count_nonzero(y[0, 0, 0]) == 1

    c = cases["repeated_writes"]
    n = len(c["k"])
    q = torch.zeros(1, 1, n, r)
    q[0, 0, :, 0] = 1.0
    k = q.clone()
    v = torch.zeros(1, 1, n, dv)
    v[0, 0, :, 0] = torch.tensor([x[0] for x in c["v"]])
    S0 = torch.zeros(1, 1, r, dv)
    S0[0, 0, 0, 0] = c["S0"][0][0]
    beta = torch.tensor(c["beta"], dtype=torch.float32).view(1, 1, n)
    y, S = _run(la, dict(q=q, k=k, v=v, beta=beta, S0=S0))
    assert list(y[0, 0, :, 0]) == [s[0][0] for s in c["S_after_each_token"]]


CASES = [
    # dtype, r, dv, T, with_state, with_beta
    (torch.float32, 128, 128, 300, True, True),
    (torch.bfloat16, 128, 128, 300, True, True),
    (torch.bfloat16, 128, 96, 65, False, True),    # three 32-column slices
    (torch.float32, 64, 64, 33, True, False),
    (torch.bfloat16, 32, 32, 31, True, True),      # one active warp of four
    (torch.float32, 256, 64, 100, True, True),     # 16-column slices
    (torch.bfloat16, 256, 32, 1, False, False),
    (torch.bfloat16, 64, 160, 97, True, True),
]


@pytest.mark.parametrize("dtype,r,dv,T,with_state,with_beta", CASES,
                         ids=[f"{str(c[0])[6:]}-r{c[1]}-dv{c[2]}-T{c[3]}-S{int(c[4])}-b{int(c[5])}" for c in CASES])
def test_delta_parity(la, oracle_mod, dtype, r, dv, T, with_state, with_beta):
    d = _inputs(2, 3, T, r, dv, dtype, with_state, with_beta, seed=81 + r + dv + T)
    y_ref, S_ref = _oracle(oracle_mod, d)
    y, S = _run(la, d)
    assert np.isfinite(y).all() and np.isfinite(S).all()
    assert_close(S, S_ref, TOL_F32, "delta S")
    assert_close(y, y_ref, TOL_F32 if dtype == torch.float32 else TOL_BF16, "delta y")


def test_delta_empty_sequence_copies_state(la):
    d = _inputs(1, 2, 0, 128, 64, torch.bfloat16, True, True, seed=90)
    y, S = _run(la, d)
    assert y.shape == (1, 2, 0, 64)
    assert np.array_equal(S, d["S0"].numpy())
    d["S0"] = None
    _, S = _run(la, d)
    assert not S.any()


def test_delta_in_place_continuation(la):
    """S0 may be S_out; and two halves chained through the state equal one call."""
    d = _inputs(1, 2, 200, 128, 128, torch.float32, True, True, seed=91)
    g = {k: v.cuda() for k, v in d.items()}
    y_full, S_full = la.delta_rule(g["q"], g["k"], g["v"], beta=g["beta"], S0=g["S0"])
    S = g["S0"].clone()
    h = 77
    y1, _ = la.delta_rule(g["q"][:, :, :h].contiguous(), g["k"][:, :, :h].contiguous(), g["v"][:, :, :h].contiguous(),
                          beta=g["beta"][:, :, :h].contiguous(), S0=S, S_out=S)
    y2, _ = la.delta_rule(g["q"][:, :, h:].contiguous(), g["k"][:, :, h:].contiguous(), g["v"][:, :, h:].contiguous(),
                          beta=g["beta"][:, :, h:].contiguous(), S0=S, S_out=S)
    assert la.last_device_status() == 0
    assert torch.equal(torch.cat([y1, y2], dim=2), y_full)
    assert torch.equal(S, S_full)


def test_delta_full_size_sampled_heads(la, oracle_mod):
    """B4 H16 T4096 r = dv = 128 BF16 (the measured shape), in the launch the
    benchmark times; the oracle recomputes three sampled heads (heads are independent)."""
    from recurrent_state_02_gb300 import workloads as W
    d = W.delta_inputs(W.DELTA)
    y, S = _run(la, d)
    for b, h in ((0, 0), (2, 7), (3, 15)):
        one = {k: v[b:b + 1, h:h + 1].contiguous() for k, v in d.items() if v is not None}
        one["S0"] = None
        y_ref, S_ref = _oracle(oracle_mod, one)
        assert_close(S[b:b + 1, h:h + 1], S_ref, TOL_F32, f"delta S head {b},{h}")
        assert_close(y[b:b + 1, h:h + 1], y_ref, TOL_BF16, f"delta y head {b},{h}")


# ---------------------------------------------------------------- chunked form
# la_delta_rule_chunked rounds the operands of its products to BF16 (S_prev,
# W = T K, T and V'), with FP32 accumulation and an FP32 state; a simulation of
# that rounding on unit keys gives about 5e-3 relative to the largest entry on
# y and S over 2048 tokens.  Both are held to 2e-2.
TOL_TC = 2e-2

TC_CASES = [
    # T, dv, H, with_state, with_beta
    (1, 64, 2, True, True),
    (63, 128, 2, False, True),
    (64, 128, 2, True, True),
    (65, 64, 3, True, False),
    (200, 192, 2, True, True),     # three 64-column slices, ragged last chunk
    (1000, 128, 1, True, True),
    (2048, 64, 1, False, False),   # beta = 1
]


def _run_tc(la, d):
    g = {k: (v.cuda() if v is not None else None) for k, v in d.items()}
    y, S = la.delta_rule_chunked(g["q"], g["k"], g["v"], beta=g["beta"], S0=g["S0"])
    assert la.last_device_status() == 0
    return y.float().cpu().numpy(), S.cpu().numpy()


@pytest.mark.parametrize("T,dv,H,with_state,with_beta", TC_CASES,
                         ids=[f"T{c[0]}-dv{c[1]}-H{c[2]}-S{int(c[3])}-b{int(c[4])}" for c in TC_CASES])
def test_delta_chunked_parity(la, oracle_mod, T, dv, H, with_state, with_beta):
    d = _inputs(2, H, T, 128, dv, torch.bfloat16, with_state, with_beta, seed=300 + T + dv)
    y_ref, S_ref = _oracle(oracle_mod, d)
    y, S = _run_tc(la, d)
    assert np.isfinite(y).all() and np.isfinite(S).all()
    assert_close(S, S_ref, TOL_TC, "chunked delta S")
    assert_close(y, y_ref, TOL_TC, "chunked delta y")


def test_delta_chunked_pages_example(la):
    """Three writes of one unit key with beta = 1/2 from S = 2 (the pages' repeated
    writes): every product is exact in BF16, so the chunked form returns the
    printed values exactly."""
    cases = {c["name"]: c for c in json.load(open(GOLDEN))["cases"]}
    c = cases["repeated_writes"]
    n, r, dv = len(c["k"]), 128, 64
    q = torch.zeros(1, 1, n, r, dtype=torch.bfloat16)
    q[0, 0, :, 0] = 1.0
    k = q.clone()
    v = torch.zeros(1, 1, n, dv, dtype=torch.bfloat16)
    v[0, 0, :, 0] = torch.tensor([x[0] for x in c["v"]], dtype=torch.bfloat16)
    S0 = torch.zeros(1, 1, r, dv)
    S0[0, 0, 0, 0] = c["S0"][0][0]
    beta = torch.tensor(c["beta"], dtype=torch.float32).view(1, 1, n)
    y, S = _run_tc(la, dict(q=q, k=k, v=v, beta=beta, S0=S0))
    assert list(y[0, 0, :, 0]) == [s[0][0] for s in c["S_after_each_token"]]
    assert S[0, 0, 0, 0] == c["S_after_each_token"][-1][0][0] and np.count_nonzero(S) == 1


def test_delta_chunked_empty_sequence_copies_state(la):
    d = _inputs(1, 2, 0, 128, 64, torch.bfloat16, True, True, seed=92)
    g = {k: v.cuda() for k, v in d.items()}
    y, S = la.delta_rule_chunked(g["q"], g["k"], g["v"], beta=g["beta"], S0=g["S0"])
    assert la.last_device_status() == 0
    assert y.shape == (1, 2, 0, 64) and torch.equal(S.cpu(), d["S0"])


def test_delta_chunked_in_place_continuation(la):
    """S0 may be S_out; split at a chunk boundary, two calls chained through the
    FP32 state give the bits of one call."""
    d = _inputs(1, 2, 300, 128, 128, torch.bfloat16, True, True, seed=93)
    g = {k: v.cuda() for k, v in d.items()}
    y_full, S_full = la.delta_rule_chunked(g["q"], g["k"], g["v"], beta=g["beta"], S0=g["S0"])
    S = g["S0"].clone()
    h = 128
    y1, _ = la.delta_rule_chunked(g["q"][:, :, :h].contiguous(), g["k"][:, :, :h].contiguous(),
                                  g["v"][:, :, :h].contiguous(), beta=g["beta"][:, :, :h].contiguous(), S0=S, S_out=S)
    y2, _ = la.delta_rule_chunked(g["q"][:, :, h:].contiguous(), g["k"][:, :, h:].contiguous(),
                                  g["v"][:, :, h:].contiguous(), beta=g["beta"][:, :, h:].contiguous(), S0=S, S_out=S)
    assert la.last_device_status() == 0
    assert torch.equal(torch.cat([y1, y2], dim=2), y_full)
    assert torch.equal(S, S_full)


def test_delta_chunked_full_size_sampled_heads(la, oracle_mod):
    """B4 H16 T4096 r = dv = 128 BF16 through the chunked kernel, in the launch the
    benchmark times; the oracle recomputes three sampled heads."""
    from recurrent_state_02_gb300 import workloads as W
    d = W.delta_inputs(W.DELTA)
    y, S = _run_tc(la, d)
    assert np.isfinite(y).all() and np.isfinite(S).all()
    for b, h in ((0, 0), (1, 9), (3, 15)):
        one = {k: v[b:b + 1, h:h + 1].contiguous() for k, v in d.items() if v is not None}
        one["S0"] = None
        y_ref, S_ref = _oracle(oracle_mod, one)
        assert_close(S[b:b + 1, h:h + 1], S_ref, TOL_TC, f"chunked delta S head {b},{h}")
        assert_close(y[b:b + 1, h:h + 1], y_ref, TOL_TC, f"chunked delta y head {b},{h}")


def test_delta_chunked_long_sequence(la, oracle_mod):
    """512 chunks (T = 32768) with a carried state: the chain's load stages,
    [-W; Q] buffers, accumulator buffers and barrier phases each wrap around
    hundreds of times; both heads against the oracle."""
    d = _inputs(1, 2, 32768, 128, 128, torch.bfloat16, True, True, seed=94)
    y, S = _run_tc(la, d)
    assert np.isfinite(y).all() and np.isfinite(S).all()
    for h in range(2):
        one = {k: (v[:, h:h + 1].contiguous() if v is not None else None) for k, v in d.items()}
        y_ref, S_ref = _oracle(oracle_mod, one)
        assert_close(S[:, h:h + 1], S_ref, TOL_TC, f"chunked delta S head {h}")
        assert_close(y[:, h:h + 1], y_ref, TOL_TC, f"chunked delta y head {h}")
