"""Precision sweep ("Linear attention：把历史写进状态", section "长历史下，状态的数值范围会增长",
its reproducible check): fixed Q/K/V, the FP64 recurrence as reference, sweep
the sequence length, the input scale and the chunk size, and record the largest
error and the smallest denominator.

The BF16 tensor-core path has a fixed chunk of 64 tokens, so the chunk axis is
swept on the oracle's chunkwise route (FP64) against its token recurrence; the
GPU is swept over T x scale x gate.  Run with -s to see the table."""
import numpy as np
import pytest
import torch

from conftest import max_rel_err, row_rel_err, to_oracle

TOL = 2e-2


@pytest.fixture(scope="module")
def la():
    from recurrent_state_02_gb300 import build
    build.build()
    import recurrent_state_02_gb300 as la_mod
    assert torch.cuda.is_available()
    return la_mod


def _min_denominator(q, k, alpha, eps):
    """Smallest phi(q_t) . z_t + eps over all tokens and heads, in FP64 (a diagnostic)."""
    phi = lambda x: np.where(x > 0, x + 1.0, np.exp(np.minimum(x, 0.0)))
    qf, kf = phi(q.float().double().numpy()), phi(k.float().double().numpy())
    B, H, T, r = qf.shape
    z = np.zeros((B, H, r))
    den_min = np.inf
    for t in range(T):
        a = alpha[:, :, t].double().numpy()[..., None] if alpha is not None else 1.0
        z = a * z + kf[:, :, t]
        den_min = min(den_min, float(np.min(np.sum(qf[:, :, t] * z, axis=-1) + eps)))
    return den_min


@pytest.mark.gpu
@pytest.mark.parametrize("gated", [False, True])
@pytest.mark.parametrize("scale", [0.5, 1.0, 2.0, 4.0])
@pytest.mark.parametrize("T", [64, 1024, 8192])
def test_precision_sweep_gpu(la, oracle_mod, T, scale, gated):
    from recurrent_state_02_gb300 import workloads as W
    w = W.Workload("sweep", B=1, H=2, T=T, dtype=torch.bfloat16, gated=gated, scale=scale, seed=71)
    inp = W.prefill_inputs(w)
    ref = oracle_mod.scan(to_oracle(inp["q"]), to_oracle(inp["k"]), to_oracle(inp["v"]), alpha=to_oracle(inp["alpha"]),
                          eps=1e-6, threads=0)
    d = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    y, S, z = la.prefill_chunked(d["q"], d["k"], d["v"], alpha=d["alpha"])
    assert la.last_device_status() == 0
    got = (y.float().cpu().numpy(), S.cpu().numpy(), z.cpu().numpy())
    errs = [max_rel_err(g, r) for g, r in zip(got, ref)]
    rows = [row_rel_err(g, r) for g, r in zip(got, ref)]
    den = _min_denominator(inp["q"], inp["k"], inp["alpha"], 1e-6)
    print(f"\nsweep T={T:5d} scale={scale:3.1f} gated={int(gated)}  max rel err y {errs[0]:.2e} "
          f"S {errs[1]:.2e} z {errs[2]:.2e}  per row y {rows[0]:.2e} S {rows[1]:.2e} z {rows[2]:.2e}  "
          f"min denominator {den:.3e}")
    assert all(np.isfinite(g).all() for g in got)
    assert max(errs) <= TOL and max(rows) <= TOL


@pytest.mark.parametrize("C", [1, 16, 64, 256])
def test_precision_sweep_chunk(oracle_mod, C):
    """Chunk size does not change the result beyond rounding: FP64 chunkwise vs token recurrence."""
    from recurrent_state_02_gb300 import workloads as W
    w = W.Workload("sweepC", B=1, H=2, T=1000, r=64, dv=64, dtype=torch.float32, gated=True, scale=2.0, seed=72)
    inp = W.prefill_inputs(w)
    args = [to_oracle(inp[n]) for n in ("q", "k", "v")]
    ref = oracle_mod.scan(*args, alpha=to_oracle(inp["alpha"]), eps=1e-6)
    got = oracle_mod.chunkwise(*args, C, alpha=to_oracle(inp["alpha"]), eps=1e-6)
    errs = [max_rel_err(g, r) for g, r in zip(got, ref)]
    print(f"\nsweep C={C:3d} (FP64 chunkwise vs recurrence)  max rel err y {errs[0]:.2e} S {errs[1]:.2e} z {errs[2]:.2e}")
    assert max(errs) < 1e-10
