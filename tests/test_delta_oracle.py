"""Pins of the FP64 delta-rule oracle (oracle.delta) to facts fixed outside it.

LA = "Linear attention：把历史写进状态" (hs-black.github.io/posts/linear-attention),
sections "Delta rule：先读旧答案，再写误差", "重复写同一个 key：累加和纠错差在哪？" and
"key 的范数决定了纠错力度".  The memory: p = S^T k, e = v - p, S <- S + beta k e^T,
and the output reads the updated memory, y = S^T q.

Every check is a function of an oracle object ``o`` so that the planted-mistake
test can run the same checks against mutated copies of the oracle."""
import json
import os

import numpy as np
import pytest

import oracle as oracle_pkg

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "delta_examples.json")
_ORACLE_SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "linattn_oracle.c")


def _cases():
    with open(GOLDEN) as f:
        return {c["name"]: c for c in json.load(f)["cases"]}


def _run(o, k, v, q=None, beta=None, S0=None):
    k = np.asarray(k, dtype=np.float64)[None, None]
    v = np.asarray(v, dtype=np.float64)[None, None]
    q = k.copy() if q is None else np.asarray(q, dtype=np.float64)[None, None]
    b = None if beta is None else np.asarray(beta, dtype=np.float64)[None, None]
    S0 = None if S0 is None else np.asarray(S0, dtype=np.float64)[None, None]
    y, S = o.delta(q, k, v, beta=b, S0=S0)
    return y[0, 0], S[0, 0]


def check_orthogonal_keys(o):
    c = _cases()["orthogonal_keys"]
    # the error the page computes: the memory's answer for k is 2, the target 5
    S0 = np.array(c["S0"], dtype=np.float64)
    k = np.array(c["k"][0], dtype=np.float64)
    assert np.allclose(np.array(c["v"][0]) - S0.T @ k, c["error_first"])
    # after the write, query each key: the written one reads 3.5, the orthogonal one 4
    for q, want in (([1, 0], c["S_final"][0]), ([0, 1], c["S_final"][1])):
        y, S = _run(o, c["k"], c["v"], q=[q], beta=c["beta"], S0=c["S0"])
        assert np.allclose(S, c["S_final"], atol=0, rtol=0)
        assert np.allclose(y[0], want, atol=0, rtol=0)


def check_repeated_writes(o):
    c = _cases()["repeated_writes"]
    y, S = _run(o, c["k"], c["v"], q=[[1]] * 3, beta=c["beta"], S0=c["S0"])
    want = [s[0][0] for s in c["S_after_each_token"]]
    assert np.array_equal(y[:, 0], want)            # y_t = S_t with q = 1: the state after each write
    assert S[0, 0] == want[-1]
    # the errors the page lists are the gaps to the target before each write
    before = [c["S0"][0][0]] + want[:-1]
    assert np.allclose([c["v"][t][0] - before[t] for t in range(3)], c["errors"])


def check_norm_factor(o):
    """One write scales the error along k by (1 - beta ||k||^2)."""
    for norm, beta, factor in _cases()["norm_factor"]["factors"]:
        k = np.array([norm, 0.0, 0.0])
        S0 = np.array([[1.0, -2.0], [0.5, 3.0], [2.0, 1.0]])
        v = np.array([5.0, -1.0])
        e0 = v - S0.T @ k
        _, S = _run(o, [k], [v], beta=[beta], S0=S0)
        e1 = v - S.T @ k
        assert np.allclose(e1, factor * e0, rtol=1e-14, atol=1e-14)


def check_hand_example(o):
    """A non-square case worked by hand from the update (r = 2, dv = 3, so that a
    transposed read or write of S cannot pass): S0 = [[1,2,3],[4,5,6]], k = [1,2],
    v = [1,1,1], beta = 0.5: p = S0^T k = [9,12,15], e = [-8,-11,-14],
    S = S0 + 0.5 k e^T = [[-3,-3.5,-4],[-4,-6,-8]], and q = [0,1] reads row 1."""
    y, S = _run(o, [[1, 2]], [[1, 1, 1]], q=[[0, 1]], beta=[0.5], S0=[[1, 2, 3], [4, 5, 6]])
    assert np.array_equal(S, [[-3, -3.5, -4], [-4, -6, -8]])
    assert np.array_equal(y[0], [-4, -6, -8])


def check_orthonormal_keys_store_values(o):
    """With orthonormal keys and beta = 1 each write stores its value exactly: the
    memory then answers every key with its value (a plain associative table)."""
    rng = np.random.default_rng(3)
    r, dv = 6, 4
    K = np.linalg.qr(rng.standard_normal((r, r)))[0][:, rng.permutation(r)].T   # rows orthonormal
    V = rng.standard_normal((r, dv))
    _, S = _run(o, K, V, beta=np.ones(r))
    assert np.allclose(S.T @ K.T, V.T, atol=1e-12)


def check_beta_zero_keeps_memory(o):
    rng = np.random.default_rng(4)
    S0 = rng.standard_normal((3, 2))
    q = rng.standard_normal((5, 3))
    y, S = _run(o, rng.standard_normal((5, 3)), rng.standard_normal((5, 2)), q=q, beta=np.zeros(5), S0=S0)
    assert np.array_equal(S, S0)
    assert np.allclose(y, q @ S0, atol=1e-14)


def check_convergence(o):
    """Repeating one (k, v) converges to S^T k = v when 0 < beta ||k||^2 < 2."""
    k = np.array([0.6, 0.8])   # unit norm
    v = np.array([2.0, -1.0, 0.5])
    m = 60
    _, S = _run(o, [k] * m, [v] * m, beta=[1.5] * m, S0=np.zeros((2, 3)))
    assert np.allclose(S.T @ k, v, atol=1e-12)


ALL_CHECKS = [(f.__name__, f) for f in (check_orthogonal_keys, check_repeated_writes, check_norm_factor,
                                         check_hand_example, check_orthonormal_keys_store_values,
                                         check_beta_zero_keeps_memory, check_convergence)]


@pytest.mark.parametrize("name,check", ALL_CHECKS, ids=[n for n, _ in ALL_CHECKS])
def test_delta_pins(name, check):
    check(oracle_pkg)


def test_delta_input_types_agree():
    """BF16 and FP32 inputs decode exactly: the same values give the same result."""
    import torch
    g = torch.Generator().manual_seed(5)
    q, k, v = (torch.randn(2, 3, 40, 16, generator=g).bfloat16() for _ in range(3))
    beta = torch.rand(2, 3, 40, generator=g).double()
    as_bits = lambda t: t.view(torch.int16).numpy().view(np.uint16)
    y1, S1 = oracle_pkg.delta(as_bits(q), as_bits(k), as_bits(v), beta=beta.numpy())
    y2, S2 = oracle_pkg.delta(*(t.float().numpy() for t in (q, k, v)), beta=beta.numpy())
    assert np.array_equal(y1, y2) and np.array_equal(S1, S2)


MUTATIONS = [
    ("error sign", "for (int j = 0; j < dv; ++j) pe[j] = decode(p->v, p->in_type, row_v + j) - pe[j];",
     "for (int j = 0; j < dv; ++j) pe[j] = decode(p->v, p->in_type, row_v + j) + pe[j];"),
    ("prediction reads S transposed", "pe[j] += S[(size_t)i * dv + j] * kt[i];",
     "pe[j] += S[(size_t)(j % r) * dv + (i % dv)] * kt[i];"),
    ("beta dropped", "S[(size_t)i * dv + j] += beta * kt[i] * pe[j];", "S[(size_t)i * dv + j] += kt[i] * pe[j];"),
    ("write skipped", "        /* write back beta * k_t e_t^T */", "        /* write back beta * k_t e_t^T */\n        if (0)"),
]


@pytest.mark.parametrize("desc,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistakes_are_caught(tmp_path, desc, old, new):
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
