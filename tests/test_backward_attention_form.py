"""The gradients of the gated recurrence written as three causal linear attentions,
checked in FP64 against the oracle's backward (oracle.backward).

LA = "Linear attention：把历史写进状态" (hs-black.github.io/posts/linear-attention),
sections "公式里的每个维度" and "加一个门：让旧记忆逐渐淡出": S_t = alpha_t S_{t-1} +
phi(k_t) v_t^T, z_t likewise, y_t = phi(q_t)^T S_t / (phi(q_t)^T z_t + eps).  The pages
give no backward.  With dn_t = dy_t / d_t, dd_t = -(dy_t . y_t) / d_t and the decay
D(s, t) = alpha_{s+1} ... alpha_t (s <= t), the chain rule gives

    dq~_t = sum_{s<=t} D(s,t) k~_s ([v_s; 1] . [dn_t; dd_t]) + D(-1,t) (S0 dn_t + dd_t z0)
    dk~_s = sum_{t>=s} D(s,t) q~_t ([v_s; 1] . [dn_t; dd_t]) + D(s,T-1) (dS_T v_s + dz_T)
    dv_s  = sum_{t>=s} D(s,t) dn_t (q~_t . k~_s)          + D(s,T-1) dS_T^T k~_s

each an unnormalised causal linear attention (the last two in reversed time) with
the operands' roles permuted: the shapes a tensor-core form of the backward would
take.  This pins that reading outside any kernel."""
import numpy as np


def _phi(x):
    return np.where(x > 0, x + 1.0, np.exp(np.minimum(x, 0.0)))


def _dphi(x):
    return np.where(x > 0, 1.0, np.exp(np.minimum(x, 0.0)))


def test_gradients_as_linear_attentions(oracle_mod):
    rng = np.random.default_rng(21)
    T, r, dv, eps = 37, 6, 5, 1e-6
    q, k = rng.standard_normal((T, r)), rng.standard_normal((T, r))
    v, dy = rng.standard_normal((T, dv)), rng.standard_normal((T, dv))
    alpha = rng.uniform(0.3, 1.0, T)
    S0, z0 = rng.standard_normal((r, dv)) * 0.3, rng.uniform(0.5, 2.0, r)
    dS_T, dz_T = rng.standard_normal((r, dv)), rng.standard_normal(r)
    e = lambda a: a[None, None]
    y, _, _ = oracle_mod.scan(e(q), e(k), e(v), alpha=e(alpha), S0=e(S0), z0=e(z0), eps=eps)
    dq_ref, dk_ref, dv_ref, _, dS0_ref, dz0_ref = oracle_mod.backward(
        e(q), e(k), e(v), e(dy), alpha=e(alpha), S0=e(S0), z0=e(z0), dS_T=e(dS_T), dz_T=e(dz_T), eps=eps)
    y = y[0, 0]

    qt, kt = _phi(q), _phi(k)
    # D[s, t] = prod alpha_{s+1..t} for s <= t; D0[t] = prod alpha_{0..t} (the start state)
    la = np.log(alpha)
    cum = np.cumsum(la)
    D = np.where(np.arange(T)[:, None] <= np.arange(T)[None, :], np.exp(cum[None, :] - cum[:, None]), 0.0)
    D0 = np.exp(cum)
    z = D.T @ kt + D0[:, None] * z0[None, :]                 # z_t
    d = np.sum(qt * z, axis=1) + eps
    dn = dy / d[:, None]
    dd = -np.sum(dy * y, axis=1) / d
    qa = np.concatenate([dn, dd[:, None]], axis=1)           # [dn_t; dd_t]
    ka = np.concatenate([v, np.ones((T, 1))], axis=1)        # [v_s; 1]
    score = ka @ qa.T                                        # [s, t] = [v_s; 1] . [dn_t; dd_t]

    dqt = (D * score).T @ kt + D0[:, None] * (dn @ S0.T + dd[:, None] * z0[None, :])
    dkt = (D * score) @ qt + D[:, T - 1][:, None] * (v @ dS_T.T + dz_T[None, :])
    dvo = (D * (kt @ qt.T)) @ dn + D[:, T - 1][:, None] * (kt @ dS_T)
    dS0 = (D0[:, None] * qt).T @ dn + D0[T - 1] * dS_T
    dz0 = (D0 * dd) @ qt + D0[T - 1] * dz_T

    def close(got, ref):
        return np.max(np.abs(got - ref)) <= 1e-10 * max(1.0, np.max(np.abs(ref)))

    assert close(_dphi(q) * dqt, dq_ref[0, 0])
    assert close(_dphi(k) * dkt, dk_ref[0, 0])
    assert close(dvo, dv_ref[0, 0])
    assert close(dS0, dS0_ref[0, 0])
    assert close(dz0, dz0_ref[0, 0])
