"""The four full-size workloads, in the launch configuration the benchmark times,
against the FP64 oracle on every (b, h) sequence: every output token and the final
state of every head, each held to the bar per tensor and per row (every token of
y, every feature row of S, the z vector of every head)."""
import numpy as np
import pytest
import torch

from conftest import assert_close, to_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def la():
    from recurrent_state_02_gb300 import build
    build.build()
    import recurrent_state_02_gb300 as la_mod
    return la_mod


def _head_groups(B, H, per):
    heads = [(b, h) for b in range(B) for h in range(H)]
    return [heads[i:i + per] for i in range(0, len(heads), per)]


@pytest.mark.parametrize("name", ["ungated", "gated", "long"])
def test_prefill_full_size(la, oracle_mod, name):
    from recurrent_state_02_gb300 import workloads as W
    w = W.WORKLOADS[name]
    inp = W.prefill_inputs(w)
    d = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    y, S, z = la.prefill_chunked(d["q"], d["k"], d["v"], alpha=d["alpha"], chunk=w.chunk, eps=w.eps)
    assert la.last_device_status() == 0
    assert torch.isfinite(y).all() and torch.isfinite(S).all() and torch.isfinite(z).all()
    y, S, z = y.cpu(), S.cpu(), z.cpu()
    del d
    torch.cuda.empty_cache()
    # all heads, a group at a time (the oracle's threads run over the heads of a group;
    # the group bounds the host memory of the FP64 outputs)
    per = max(1, min(w.B * w.H, (1 << 27) // (w.T * w.dv)))
    worst = {"y": 0.0, "S": 0.0, "z": 0.0}
    for grp in _head_groups(w.B, w.H, per):
        sel = lambda t: None if t is None else torch.stack([t[b, h] for b, h in grp])[None]
        ref = oracle_mod.scan(to_oracle(sel(inp["q"])), to_oracle(sel(inp["k"])), to_oracle(sel(inp["v"])),
                              alpha=to_oracle(sel(inp["alpha"])), eps=w.eps)
        got = (sel(y).float().numpy(), sel(S).numpy(), sel(z).numpy())
        for what, g, r in zip(("y", "S", "z"), got, ref):
            _, r_err = assert_close(g, r, 2e-2, f"{name} {what} heads {grp[0]}..{grp[-1]}")
            worst[what] = max(worst[what], r_err)
    print(f"[parity] {name}: worst per-row error over all {w.B * w.H} heads: {worst}")


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
        assert_close(g, r, 2e-2, f"decode {what}")
