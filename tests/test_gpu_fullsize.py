"""The four full-size workloads, in the launch configuration the benchmark times,
against the FP64 oracle on sampled (b, h) sequences (every output and the final
state of each sampled sequence; all heads for decode)."""
import numpy as np
import pytest
import torch

from conftest import max_rel_err, to_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def la():
    from recurrent_state_02_gb300 import build
    build.build()
    import recurrent_state_02_gb300 as la_mod
    return la_mod


def _sample_heads(B, H):
    picks = {(0, 0), (B - 1, H - 1), (B // 2, H // 2)}
    return sorted(picks)


@pytest.mark.parametrize("name", ["ungated", "gated", "long"])
def test_prefill_full_size(la, oracle_mod, name):
    from recurrent_state_02_gb300 import workloads as W
    w = W.WORKLOADS[name]
    inp = W.prefill_inputs(w)
    d = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    y, S, z = la.prefill_chunked(d["q"], d["k"], d["v"], alpha=d["alpha"], chunk=w.chunk, eps=w.eps)
    assert la.last_device_status() == 0
    assert torch.isfinite(y).all() and torch.isfinite(S).all() and torch.isfinite(z).all()
    heads = _sample_heads(w.B, w.H)
    sel = lambda t: None if t is None else torch.stack([t[b, h] for b, h in heads])[None]
    ref_y, ref_S, ref_z = oracle_mod.scan(to_oracle(sel(inp["q"])), to_oracle(sel(inp["k"])),
                                          to_oracle(sel(inp["v"])), alpha=to_oracle(sel(inp["alpha"])), eps=w.eps)
    got_y = torch.stack([y[b, h] for b, h in heads]).float().cpu().numpy()[None]
    got_S = torch.stack([S[b, h] for b, h in heads]).cpu().numpy()[None]
    got_z = torch.stack([z[b, h] for b, h in heads]).cpu().numpy()[None]
    for what, g, r in (("y", got_y, ref_y), ("S", got_S, ref_S), ("z", got_z, ref_z)):
        err = max_rel_err(g, r)
        assert err <= 2e-2, f"{name} {what}: max rel err {err:.3e}"


def test_decode_full_size(la, oracle_mod):
    from recurrent_state_02_gb300 import workloads as W
    w = W.DECODE
    inp = W.decode_inputs(w)
    ref_y, ref_S, ref_z = oracle_mod.scan(to_oracle(inp["q"]), to_oracle(inp["k"]), to_oracle(inp["v"]),
                                          S0=to_oracle(inp["S"]), z0=to_oracle(inp["z"]), eps=w.eps)
    d = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    y = la.decode_step(d["q"], d["k"], d["v"], d["S"], d["z"], alpha=d["alpha"], eps=w.eps)
    assert la.last_device_status() == 0
    for what, g, r in (("y", y.float().cpu().numpy(), ref_y), ("S", d["S"].cpu().numpy(), ref_S),
                       ("z", d["z"].cpu().numpy(), ref_z)):
        err = max_rel_err(g, r)
        assert err <= 2e-2, f"decode {what}: max rel err {err:.3e}"
