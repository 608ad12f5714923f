"""Pins of the FP64 oracle to facts fixed outside the oracle itself.

Sources (cited by page title and section):
  LA = "Linear attention：把历史写进状态" (hs-black.github.io/posts/linear-attention)
  LC = "45. Linear Attention and Recurrent State | 线性注意力与递推状态" (datawhalechina, ch. 45)

Every check below is a plain function of an oracle object ``o`` (with
.scan/.dense/.chunkwise) so that ``test_planted_mistakes_are_caught`` can run
the same checks against copies of the oracle with a mistake planted in them.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle as oracle_pkg

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")
PHI = {"identity": oracle_pkg.PHI_IDENTITY, "relu1": oracle_pkg.PHI_RELU1, "elu1": oracle_pkg.PHI_ELU1}
ROUTES = ("scan", "dense", "chunk1", "chunk2", "chunk3")


def _cases():
    with open(GOLDEN) as f:
        return {c["name"]: c for c in json.load(f)["cases"]}


def _as4(a):
    a = np.asarray(a, dtype=np.float64)
    return a.reshape((1, 1) + a.shape)


def _run(o, route, q, k, v, **kw):
    if route == "scan":
        return o.scan(q, k, v, **kw)
    if route == "dense":
        return o.dense(q, k, v, **kw)
    return o.chunkwise(q, k, v, int(route[5:]), **kw)


def _frac(x):
    return float(Fraction(x[0], x[1]))


def _rng(seed):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------- worked examples

def check_worked_example(o, name, route):
    c = _cases()[name]
    q, k, v = _as4(c["q"]), _as4(c["k"]), _as4(c["v"])
    alpha = np.asarray(c["alpha"]).reshape(1, 1, -1) if "alpha" in c else None
    phi = PHI[c["phi"]]
    T = q.shape[2]
    y, S, z = _run(o, route, q, k, v, alpha=alpha, eps=c["eps"], phi=phi)
    if "S_final" in c:
        np.testing.assert_allclose(S[0, 0], np.asarray(c["S_final"], float), rtol=0, atol=1e-12)
    if "z_final" in c:
        np.testing.assert_allclose(z[0, 0], np.asarray(c["z_final"], float), rtol=0, atol=1e-12)
    if "S_after_each_token" in c:
        for t in range(T):
            a_t = None if alpha is None else alpha[:, :, : t + 1]
            _, St, zt = _run(o, route, q[:, :, : t + 1], k[:, :, : t + 1], v[:, :, : t + 1],
                             alpha=a_t, eps=c["eps"], phi=phi)
            np.testing.assert_allclose(St[0, 0], np.asarray(c["S_after_each_token"][t], float), atol=1e-12)
            np.testing.assert_allclose(zt[0, 0], np.asarray(c["z_after_each_token"][t], float), atol=1e-12)
    if "y_last_exact" in c:
        want = np.array([_frac(x) for x in c["y_last_exact"]])
        np.testing.assert_allclose(y[0, 0, -1], want, rtol=1e-14, atol=0)
    if "y_exact" in c:
        want = np.array([[_frac(x) for x in row] for row in c["y_exact"]])
        np.testing.assert_allclose(y[0, 0], want, rtol=1e-14, atol=0)
    if "numerator_last" in c:
        # with eps = 0 the output times the denominator is the numerator
        np.testing.assert_allclose(y[0, 0, -1] * c["denominator_last"], np.asarray(c["numerator_last"], float),
                                   rtol=1e-14)
        qf = np.asarray(c["q"], float)[-1]
        np.testing.assert_allclose(qf @ z[0, 0], c["denominator_last"], rtol=1e-14)
    if "history_weights" in c:
        # y is the weighted mean of the values with the printed weights
        w = np.asarray(c["history_weights"])
        vals = np.asarray(c["v"], float)[:, 0]
        np.testing.assert_allclose(y[0, 0, -1, 0], (w @ vals) / w.sum(), rtol=1e-14)


def check_epsilon_convention(o, route):
    c = _cases()["epsilon_convention"]
    for eps, want, tol in c["eps_cases"]:
        y, _, _ = _run(o, route, _as4(c["q"]), _as4(c["k"]), _as4(c["v"]), eps=eps, phi=oracle_pkg.PHI_IDENTITY)
        assert abs(y[0, 0, 0, 0] - want) <= tol, (eps, y[0, 0, 0, 0], want)


def check_lc_fixture_contract(o, route):
    """LC Step 4 tests: shapes, finite outputs, positive normaliser, prefix causality."""
    c = _cases()["lc_fixture_relu1"]
    q, k, v = _as4(c["q"]), _as4(c["k"]), _as4(c["v"])
    y, S, z = _run(o, route, q, k, v, eps=0.0, phi=oracle_pkg.PHI_RELU1)
    assert y.shape[2:] == (3, 1) and S.shape[2:] == (2, 1) and z.shape[2:] == (2,)
    assert np.isfinite(y).all() and (z > 0).all()
    k2, v2 = k.copy(), v.copy()
    k2[0, 0, -1] += 100.0
    v2[0, 0, -1] += 100.0
    y2, _, _ = _run(o, route, q, k2, v2, eps=0.0, phi=oracle_pkg.PHI_RELU1)
    np.testing.assert_array_equal(y[0, 0, :-1], y2[0, 0, :-1])


# ------------------------------------------------------------------- invariants

def check_repeat_invariant(o, route):
    """LA '没有 z，输出会随重复次数增长': the same (k, v) written m times reads back v."""
    r_ = _rng(1)
    m, r, dv = 7, 5, 3
    q = _as4(r_.normal(size=(m, r)))
    k = _as4(np.repeat(r_.normal(size=(1, r)), m, axis=0))
    v = _as4(np.repeat(r_.normal(size=(1, dv)), m, axis=0))
    y, _, _ = _run(o, route, q, k, v, eps=0.0)
    np.testing.assert_allclose(y[0, 0], np.repeat(v[0, 0, :1], m, axis=0), rtol=1e-13)


def check_prefix_causality(o, route):
    """LC test_prefix_causality, ELU+1 and gated: later tokens never change earlier outputs."""
    r_ = _rng(2)
    T, r, dv = 9, 4, 3
    q, k, v = (_as4(r_.normal(size=(T, n))) for n in (r, r, dv))
    alpha = r_.uniform(0.2, 1.0, size=(1, 1, T))
    y, _, _ = _run(o, route, q, k, v, alpha=alpha)
    for t in range(T):
        k2, v2, a2 = k.copy(), v.copy(), alpha.copy()
        k2[0, 0, t:] += 100.0
        v2[0, 0, t:] -= 50.0
        a2[0, 0, t:] = 0.3
        y2, _, _ = _run(o, route, q, k2, v2, alpha=a2)
        np.testing.assert_array_equal(y[0, 0, :t], y2[0, 0, :t])


def check_feature_maps(o, route):
    """With one token and a zero initial state, z_T equals phi(k) exactly: compare
    ELU+1 with the textbook ELU built from numpy's expm1, relu+1 and identity."""
    x = np.array([-100.0, -20.0, -1.5, -1.0, -1e-8, 0.0, 1e-300, 1e-8, 0.5, 1.0, 3.0, 88.0])
    r = x.size
    q = _as4(np.ones((1, r)))
    k = _as4(x[None, :])
    v = _as4(np.ones((1, 1)))
    want = {
        oracle_pkg.PHI_ELU1: np.where(x > 0, x, np.expm1(x)) + 1.0,
        oracle_pkg.PHI_RELU1: np.maximum(x, 0.0) + 1.0,
        oracle_pkg.PHI_IDENTITY: x,
    }
    # (expm1(x) + 1 rounds at the scale of 1, hence the absolute tolerance of half an ulp of 1)
    for phi, w in want.items():
        _, S, z = _run(o, route, q, k, v, eps=0.0, phi=phi)
        np.testing.assert_allclose(z[0, 0], w, rtol=1e-15, atol=2**-53)
        np.testing.assert_allclose(S[0, 0, :, 0], w, rtol=1e-15, atol=2**-53)
        if phi == oracle_pkg.PHI_ELU1:
            assert (z > 0).all()  # LC TODO 1 contract: strictly positive features


def check_single_token_closed_form(o, route):
    """T = 1: y = (q~.k~) v / (q~.k~ + eps) and S = k~ v^T, z = k~."""
    r_ = _rng(3)
    r, dv = 6, 4
    q, k, v = (_as4(r_.normal(size=(1, n))) for n in (r, r, dv))
    phi = lambda a: np.where(a > 0, a + 1.0, np.exp(a))
    qk = phi(q[0, 0, 0]) @ phi(k[0, 0, 0])
    eps = 1e-3
    y, S, z = _run(o, route, q, k, v, eps=eps)
    np.testing.assert_allclose(y[0, 0, 0], qk * v[0, 0, 0] / (qk + eps), rtol=1e-14)
    np.testing.assert_allclose(S[0, 0], np.outer(phi(k[0, 0, 0]), v[0, 0, 0]), rtol=1e-15)


def check_equal_keys_mean(o, route):
    """All keys equal and ungated, eps = 0: every weight is the same, so y_t is the running
    mean of v_1..v_t; with a constant gate a it is the mean weighted by a^(t-s)."""
    r_ = _rng(4)
    T, r, dv = 11, 3, 2
    q = _as4(r_.normal(size=(T, r)))
    k = _as4(np.repeat(r_.normal(size=(1, r)), T, axis=0))
    v = _as4(r_.normal(size=(T, dv)))
    y, _, _ = _run(o, route, q, k, v, eps=0.0)
    running = np.cumsum(v[0, 0], axis=0) / np.arange(1, T + 1)[:, None]
    np.testing.assert_allclose(y[0, 0], running, rtol=1e-13)
    a = 0.7
    yg, _, _ = _run(o, route, q, k, v, alpha=np.full((1, 1, T), a), eps=0.0)
    for t in range(T):
        w = a ** (t - np.arange(t + 1))
        np.testing.assert_allclose(yg[0, 0, t], (w @ v[0, 0, : t + 1]) / w.sum(), rtol=1e-13)


def check_zero_gate_forgets(o, route):
    """alpha_t = 0 erases everything written before t (and the carried state)."""
    r_ = _rng(5)
    T, r, dv = 8, 4, 3
    q, k, v = (_as4(r_.normal(size=(T, n))) for n in (r, r, dv))
    alpha = r_.uniform(0.5, 1.0, size=(1, 1, T))
    alpha[0, 0, 5] = 0.0
    S0 = r_.normal(size=(1, 1, r, dv))
    z0 = r_.uniform(1, 2, size=(1, 1, r))
    y, S, z = _run(o, route, q, k, v, alpha=alpha, S0=S0, z0=z0)
    al = alpha[:, :, 5:].copy()
    al[0, 0, 0] = 1.0
    y_tail, S_tail, z_tail = _run(o, route, q[:, :, 5:], k[:, :, 5:], v[:, :, 5:], alpha=al)
    np.testing.assert_allclose(y[0, 0, 5:], y_tail[0, 0], rtol=1e-13)
    np.testing.assert_allclose(S, S_tail, rtol=1e-13)
    np.testing.assert_allclose(z, z_tail, rtol=1e-13)


def check_value_linearity(o, route):
    """y and S are linear in v (q, k, gates fixed); z does not depend on v."""
    r_ = _rng(6)
    T, r, dv = 10, 4, 3
    q, k = (_as4(r_.normal(size=(T, r))) for _ in range(2))
    v1, v2 = (_as4(r_.normal(size=(T, dv))) for _ in range(2))
    alpha = r_.uniform(0.3, 1.0, size=(1, 1, T))
    y1, S1, z1 = _run(o, route, q, k, v1, alpha=alpha)
    y2, S2, z2 = _run(o, route, q, k, v2, alpha=alpha)
    y3, S3, z3 = _run(o, route, q, k, 2.0 * v1 - 3.0 * v2, alpha=alpha)
    np.testing.assert_allclose(y3, 2 * y1 - 3 * y2, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(S3, 2 * S1 - 3 * S2, rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(z1, z3)


def check_rectangular_state_layout(o, route):
    """r != dv pins the orientation of S (rows = feature index, columns = value index):
    S_T = sum_t phi(k_t) v_t^T computed by hand, and y read as phi(q)^T S / phi(q)^T z."""
    r_ = _rng(7)
    T, r, dv = 5, 3, 7
    q, k, v = _as4(r_.normal(size=(T, r))), _as4(r_.normal(size=(T, r))), _as4(r_.normal(size=(T, dv)))
    phi = lambda a: np.where(a > 0, a + 1.0, np.exp(a))
    Kf, Qf, V = phi(k[0, 0]), phi(q[0, 0]), v[0, 0]
    y, S, z = _run(o, route, q, k, v, eps=0.0)
    S_hand = sum(np.outer(Kf[t], V[t]) for t in range(T))
    np.testing.assert_allclose(S[0, 0], S_hand, rtol=1e-13)
    np.testing.assert_allclose(z[0, 0], Kf.sum(0), rtol=1e-13)
    np.testing.assert_allclose(y[0, 0, -1], (Qf[-1] @ S_hand) / (Qf[-1] @ Kf.sum(0)), rtol=1e-13)


def check_bf16_decoding(o, route):
    """BF16 inputs travel as raw bits: 0x3F80 = 1, 0xC000 = -2, 0x3F00 = 0.5, 0x4049 = 3.140625."""
    bits = np.array([0x3F80, 0xC000, 0x3F00, 0x4049], dtype=np.uint16)
    vals = np.array([1.0, -2.0, 0.5, 3.140625])
    k = bits.reshape(1, 1, 1, 4)
    q = np.full((1, 1, 1, 4), 0x3F80, dtype=np.uint16)
    v = np.full((1, 1, 1, 1), 0x3F80, dtype=np.uint16)
    _, _, z = _run(o, route, q, k, v, eps=0.0, phi=oracle_pkg.PHI_IDENTITY)
    np.testing.assert_array_equal(z[0, 0], vals)


ALL_CHECKS = [
    *(("worked:" + n, (lambda n: lambda o, rt: check_worked_example(o, n, rt))(n))
      for n in ("accumulators_scalar_value", "matrix_value", "exercise_1", "forget_gate_half",
                "exercise_2", "lc_fixture_relu1")),
    ("epsilon", check_epsilon_convention),
    ("lc_contract", check_lc_fixture_contract),
    ("repeat", check_repeat_invariant),
    ("causality", check_prefix_causality),
    ("feature_maps", check_feature_maps),
    ("single_token", check_single_token_closed_form),
    ("equal_keys", check_equal_keys_mean),
    ("zero_gate", check_zero_gate_forgets),
    ("linearity", check_value_linearity),
    ("layout", check_rectangular_state_layout),
    ("bf16", check_bf16_decoding),
]


@pytest.mark.parametrize("route", ROUTES)
@pytest.mark.parametrize("name,check", ALL_CHECKS, ids=[n for n, _ in ALL_CHECKS])
def test_pin(oracle_mod, name, check, route):
    check(oracle_mod, route)


# --------------------------------------------- the three routes agree (random) --

@pytest.mark.parametrize("gated", [False, True])
@pytest.mark.parametrize("with_state", [False, True])
def test_dense_equals_scan(oracle_mod, gated, with_state):
    r_ = _rng(10 + 2 * gated + with_state)
    B, H, T, r, dv = 2, 3, 19, 5, 6
    q, k = (r_.normal(size=(B, H, T, r)) for _ in range(2))
    v = r_.normal(size=(B, H, T, dv))
    alpha = r_.uniform(0.05, 1.0, size=(B, H, T)) if gated else None
    S0 = r_.normal(size=(B, H, r, dv)) if with_state else None
    z0 = r_.uniform(1, 100, size=(B, H, r)) if with_state else None
    a = oracle_mod.scan(q, k, v, alpha=alpha, S0=S0, z0=z0)
    b = oracle_mod.dense(q, k, v, alpha=alpha, S0=S0, z0=z0)
    for x, y_ in zip(a, b):
        np.testing.assert_allclose(x, y_, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("C", [1, 3, 16, 64, 100, 131])
@pytest.mark.parametrize("gated", [False, True])
def test_chunkwise_equals_scan(oracle_mod, C, gated):
    """LA '动手实验': changing the chunk size must not change the result."""
    r_ = _rng(20 + C + gated)
    B, H, T, r, dv = 1, 2, 131, 8, 5
    q, k = (r_.normal(size=(B, H, T, r)) for _ in range(2))
    v = r_.normal(size=(B, H, T, dv))
    alpha = r_.uniform(0.05, 1.0, size=(B, H, T)) if gated else None
    if gated:
        alpha[0, 1, 40] = 0.0
    S0 = r_.normal(size=(B, H, r, dv))
    z0 = r_.uniform(1, 100, size=(B, H, r))
    a = oracle_mod.scan(q, k, v, alpha=alpha, S0=S0, z0=z0)
    b = oracle_mod.chunkwise(q, k, v, C, alpha=alpha, S0=S0, z0=z0)
    for x, y_ in zip(a, b):
        np.testing.assert_allclose(x, y_, rtol=1e-11, atol=1e-12)


def test_continuation_and_threads(oracle_mod):
    """Prefill of T1 then T2 tokens from the returned state equals one prefill of T1+T2
    (the state is the checkpoint), bit for bit; the thread count changes nothing."""
    r_ = _rng(30)
    B, H, T, r, dv = 2, 2, 40, 6, 5
    q, k = (r_.normal(size=(B, H, T, r)).astype(np.float32) for _ in range(2))
    v = r_.normal(size=(B, H, T, dv)).astype(np.float32)
    alpha = r_.uniform(0.5, 1.0, size=(B, H, T))
    y, S, z = oracle_mod.scan(q, k, v, alpha=alpha, threads=1)
    y4, S4, z4 = oracle_mod.scan(q, k, v, alpha=alpha, threads=4)
    np.testing.assert_array_equal(y, y4)
    t1 = 17
    ya, Sa, za = oracle_mod.scan(q[:, :, :t1], k[:, :, :t1], v[:, :, :t1], alpha=alpha[:, :, :t1])
    yb, Sb, zb = oracle_mod.scan(q[:, :, t1:], k[:, :, t1:], v[:, :, t1:], alpha=alpha[:, :, t1:], S0=Sa, z0=za)
    np.testing.assert_array_equal(np.concatenate([ya, yb], axis=2), y)
    np.testing.assert_array_equal(Sb, S)
    np.testing.assert_array_equal(zb, z)
    ones, _, _ = oracle_mod.scan(q, k, v, alpha=np.ones((B, H, T)))
    none, _, _ = oracle_mod.scan(q, k, v)
    np.testing.assert_array_equal(ones, none)


def test_oracle_rejects_bad_arguments(oracle_mod):
    """LC test_input_contract: an empty sequence is rejected."""
    e = np.empty((1, 1, 0, 2))
    with pytest.raises(ValueError):
        oracle_mod.scan(e, e, np.empty((1, 1, 0, 1)))
    with pytest.raises(ValueError):
        oracle_mod.scan(np.ones((1, 1, 2, 2)), np.ones((1, 1, 2, 3)), np.ones((1, 1, 2, 1)))


# ------------------------------------------- planted mistakes must be caught --

_ORACLE_SRC = os.path.join(os.path.dirname(oracle_pkg.__file__), "linattn_oracle.c")

# (description, text in the oracle, replacement) -- each a plausible slip.
MUTATIONS = [
    ("feature map sign", "return x > 0.0 ? x + 1.0 : exp(x);", "return x > 0.0 ? x + 1.0 : exp(-x);"),
    ("ELU branch off by one", "return x > 0.0 ? x + 1.0 : exp(x);", "return x > 0.0 ? x : exp(x);"),
    ("gate dropped on S", "Si[j] = a * Si[j] + kt[i]", "Si[j] = Si[j] + kt[i]"),
    ("gate dropped on z", "z[i] = a * z[i] + kt[i];", "z[i] = z[i] + kt[i];"),
    ("eps as a floor", "num[j] / (den + p->eps)", "num[j] / (den > p->eps ? den : p->eps)"),
    ("normaliser dropped", "num[j] / (den + p->eps)", "num[j] / (1.0 + p->eps)"),
    ("state read transposed", "num[j] += qt[i] * Si[j];", "num[j] += qt[i] * S[(size_t)j * dv + (i % dv)];"),
    ("key and query swapped in the write",
     "kt[i] = phi(decode(p->k, p->in_type, row_qk + i), p->phi_kind);",
     "kt[i] = phi(decode(p->q, p->in_type, row_qk + i), p->phi_kind);"),
    ("read before write", "        /* y_t = phi(q_t)^T S_t / (phi(q_t)^T z_t + eps) */",
     "        continue; /* moved */"),
]


@pytest.mark.parametrize("desc,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistakes_are_caught(tmp_path, desc, old, new):
    src = open(_ORACLE_SRC).read()
    assert old in src, f"mutation anchor missing: {old}"
    if desc == "read before write":
        # move the read of y_t above the state update: emit the output from the previous state
        src = src.replace(
            "        /* S_t = a S_{t-1} + phi(k_t) v_t^T ;  z_t = a z_{t-1} + phi(k_t) */",
            "        { double den = 0.0; for (int j = 0; j < dv; ++j) num[j] = 0.0;\n"
            "          for (int i = 0; i < r; ++i) { const double *Si = S + (size_t)i * dv;\n"
            "            for (int j = 0; j < dv; ++j) num[j] += qt[i] * Si[j]; den += qt[i] * z[i]; }\n"
            "          for (int j = 0; j < dv; ++j) p->y[row_v + j] = num[j] / (den + p->eps); }\n"
            "        /* S_t = a S_{t-1} + phi(k_t) v_t^T ;  z_t = a z_{t-1} + phi(k_t) */")
        src = src.replace(old, "        if (1) continue;\n" + old)
    else:
        src = src.replace(old, new)
    path = tmp_path / "mutant.c"
    path.write_text(src)
    lib = oracle_pkg.build(force=True, src=str(path), out=str(tmp_path / "libmutant.so"))
    mutant = oracle_pkg.variant(lib)
    caught = []
    for name, check in ALL_CHECKS:
        try:
            check(mutant, "scan")
        except (AssertionError, ValueError, FloatingPointError):
            caught.append(name)
    assert caught, f"no pin catches the planted mistake: {desc}"
