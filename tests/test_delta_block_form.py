"""The chunk form of the delta rule used by la_delta_rule_chunked, checked in FP64
against the token recurrence of the oracle (oracle.delta).

LA = "Linear attention：把历史写进状态" (hs-black.github.io/posts/linear-attention),
section "Delta rule：先读旧答案，再写误差": per token, p = S^T k, S <- S + beta k (v - p)^T,
y = S^T q after the write.  The pages say that a block form needs its own algorithm
and give none (section "训练时，状态更新也能按块并行").  The one the kernels use follows
from the update: for a chunk with rows K, Q, V and the state S_prev before it, the
written rows V' = beta (V - K S) solve

    (I + L) V' = diag(beta) X,   X = V - K S_prev,   L = diag(beta) strictly-lower(K K^T),

so V' = T X with T = (I + L)^-1 diag(beta), S_next = S_prev + K^T V' and
Y = Q S_prev + ((Q K^T) . M) V' (M causal with its diagonal).  The per-chunk kernel
forms T by blocks: the diagonal blocks by forward substitution, the lower block of
a 2 x 2 split as -T11 (K1 K0^T) T00.

The chain kernel takes the state-independent products first: with W = T K and
U = T V, V' = U - W S_prev.

These tests write that algebra out in numpy (FP64) and hold it to the oracle,
so that the reading the GPU path rests on is pinned outside the GPU path."""
import numpy as np
import pytest


def _chunk_form(q, k, v, beta, S0, C):
    """The chunk equations above for one (b, h): q, k [T, r], v [T, dv], beta [T]."""
    T = q.shape[0]
    S = S0.copy()
    y = np.empty((T, v.shape[1]))
    for t0 in range(0, T, C):
        Q, K, V, b = q[t0:t0 + C], k[t0:t0 + C], v[t0:t0 + C], beta[t0:t0 + C]
        n = K.shape[0]
        L = np.tril(b[:, None] * (K @ K.T), -1)
        Tm = np.linalg.solve(np.eye(n) + L, np.diag(b))
        Vp = Tm @ (V - K @ S)
        y[t0:t0 + n] = Q @ S + np.tril(Q @ K.T) @ Vp
        S = S + K.T @ Vp
    return y, S


def _chunk_form_wu(q, k, v, beta, S0, C):
    """The same chunk with the state-independent products taken first, as the
    chain kernel forms them: W = T K and U = T V, then one stacked product
    [U; 0] + [-W; Q] S_prev gives [V'; Q S_prev], and [0; A] V' adds the
    in-chunk reads to the lower half."""
    T = q.shape[0]
    S = S0.copy()
    y = np.empty((T, v.shape[1]))
    for t0 in range(0, T, C):
        Q, K, V, b = q[t0:t0 + C], k[t0:t0 + C], v[t0:t0 + C], beta[t0:t0 + C]
        n = K.shape[0]
        L = np.tril(b[:, None] * (K @ K.T), -1)
        Tm = np.linalg.solve(np.eye(n) + L, np.diag(b))
        W, U = Tm @ K, Tm @ V
        D = np.vstack([U, np.zeros((n, V.shape[1]))]) + np.vstack([-W, Q]) @ S
        Vp = D[:n]
        A = np.tril(Q @ K.T)
        D = D + np.vstack([np.zeros((n, n)), A]) @ Vp
        y[t0:t0 + n] = D[n:]
        S = S + K.T @ Vp
    return y, S


def _forward_substitution(L, b):
    """(I + L)^-1 diag(b) for strictly lower L, column by column, each finished row
    subtracted from the rows below it (the order of the per-chunk kernel)."""
    n = L.shape[0]
    T = np.zeros((n, n))
    for j in range(n):
        acc = np.zeros(n)
        acc[j] = b[j]
        for u in range(n - 1):
            acc[u + 1:] -= L[u + 1:, u] * acc[u]
        T[:, j] = acc
    return T


def _inputs(rng, T, r, dv, unit=True):
    q = rng.standard_normal((T, r))
    k = rng.standard_normal((T, r))
    if unit:
        q /= np.linalg.norm(q, axis=1, keepdims=True)
        k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = rng.standard_normal((T, dv))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal(T)))
    S0 = rng.standard_normal((r, dv)) * 0.1
    return q, k, v, beta, S0


@pytest.mark.parametrize("T,C", [(1, 64), (63, 64), (64, 64), (200, 64), (130, 16), (97, 1), (150, 256)])
def test_chunk_form_equals_token_recurrence(oracle_mod, T, C):
    rng = np.random.default_rng(1000 + T + C)
    q, k, v, beta, S0 = _inputs(rng, T, 24, 16)
    y_ref, S_ref = oracle_mod.delta(q[None, None], k[None, None], v[None, None], beta=beta[None, None],
                                    S0=S0[None, None])
    y, S = _chunk_form(q, k, v, beta, S0, C)
    assert np.max(np.abs(y - y_ref[0, 0])) <= 1e-12 * np.max(np.abs(y_ref))
    assert np.max(np.abs(S - S_ref[0, 0])) <= 1e-12 * np.max(np.abs(S_ref))


@pytest.mark.parametrize("T,C", [(1, 64), (64, 64), (200, 64), (97, 16)])
def test_precomputed_products_form_equals_token_recurrence(oracle_mod, T, C):
    rng = np.random.default_rng(2000 + T + C)
    q, k, v, beta, S0 = _inputs(rng, T, 24, 16)
    y_ref, S_ref = oracle_mod.delta(q[None, None], k[None, None], v[None, None], beta=beta[None, None],
                                    S0=S0[None, None])
    y, S = _chunk_form_wu(q, k, v, beta, S0, C)
    assert np.max(np.abs(y - y_ref[0, 0])) <= 1e-12 * np.max(np.abs(y_ref))
    assert np.max(np.abs(S - S_ref[0, 0])) <= 1e-12 * np.max(np.abs(S_ref))


def test_chunk_form_special_cases(oracle_mod):
    """beta = 0 writes nothing (the state and the reads of it are unchanged), a
    repeated unit key with beta = 1 stores the last value exactly, and a zero
    key row (a padded token) leaves the chunk's other writes as they are."""
    rng = np.random.default_rng(7)
    q, k, v, beta, S0 = _inputs(rng, 40, 8, 4)
    y, S = _chunk_form(q, k, v, np.zeros(40), S0, 16)
    assert np.allclose(S, S0, rtol=0, atol=0) and np.allclose(y, q @ S0, rtol=1e-14, atol=1e-14)

    kk = np.zeros((5, 8))
    kk[:, 2] = 1.0
    vv = rng.standard_normal((5, 4))
    y, S = _chunk_form(kk, kk, vv, np.ones(5), np.zeros((8, 4)), 64)
    assert np.allclose(S[2], vv[-1], rtol=0, atol=1e-14) and np.allclose(y, vv, rtol=0, atol=1e-14)

    k2 = k.copy()
    k2[10] = 0.0
    y_ref, S_ref = oracle_mod.delta(q[None, None], k2[None, None], v[None, None], beta=beta[None, None],
                                    S0=S0[None, None])
    y, S = _chunk_form(q, k2, v, beta, S0, 16)
    assert np.max(np.abs(y - y_ref[0, 0])) <= 1e-12 * np.max(np.abs(y_ref))
    assert np.max(np.abs(S - S_ref[0, 0])) <= 1e-12 * np.max(np.abs(S_ref))


@pytest.mark.parametrize("zero_tail", [0, 19])
def test_two_by_two_block_inverse(zero_tail):
    """T = (I + L)^-1 diag(beta) of a 64-token chunk by blocks of 32: the diagonal
    blocks by forward substitution, T10 = -T11 (K1 K0^T) T00 with the raw key
    products.  Padded tokens (beta = 0, zero keys) give zero rows and columns."""
    rng = np.random.default_rng(11 + zero_tail)
    K = rng.standard_normal((64, 128))
    K /= np.linalg.norm(K, axis=1, keepdims=True)
    b = 1.0 / (1.0 + np.exp(-rng.standard_normal(64)))
    if zero_tail:
        K[64 - zero_tail:] = 0.0
        b[64 - zero_tail:] = 0.0
    G = K @ K.T
    L = np.tril(b[:, None] * G, -1)
    direct = np.linalg.solve(np.eye(64) + L, np.diag(b))
    T00 = _forward_substitution(L[:32, :32], b[:32])
    T11 = _forward_substitution(L[32:, 32:], b[32:])
    T10 = -T11 @ G[32:, :32] @ T00
    blocks = np.block([[T00, np.zeros((32, 32))], [T10, T11]])
    assert np.max(np.abs(blocks - direct)) <= 1e-13
    if zero_tail:
        assert not blocks[64 - zero_tail:].any() and not blocks[:, 64 - zero_tail:].any()
