"""la_prefill_chunked_noalloc (scratch compiled into the library) against
la_prefill_chunked with a caller workspace: the same kernels and the same plan,
so the results are bit-identical.  Two calls in a row reuse the one buffer.
This file runs last and depends on nothing the other tests leave behind."""
import pytest
import torch

pytestmark = pytest.mark.gpu

SEG_T = 47 * 64 - 21   # few heads and 47 chunks: the sequence is split into segments


@pytest.fixture(scope="module")
def la():
    from recurrent_state_02_gb300 import build
    build.build()
    import recurrent_state_02_gb300 as la_mod
    assert torch.cuda.is_available()
    return la_mod


def _inputs(B, H, T, gated, seed):
    from recurrent_state_02_gb300 import workloads as W
    w = W.Workload("noalloc", B=B, H=H, T=T, dtype=torch.bfloat16, gated=gated, seed=seed)
    return {k: (v.cuda() if v is not None else None) for k, v in W.prefill_inputs(w, with_state=True).items()}


def _outputs(d):
    B, H, T, dv = d["v"].shape
    r = d["q"].shape[3]
    return (torch.empty_like(d["v"]), torch.empty(B, H, r, dv, device="cuda"),
            torch.empty(B, H, r, device="cuda"))


def test_noalloc_matches_workspace_entry_point(la):
    assert la.prefill_workspace_bytes(1, 3, SEG_T, 128, 128) > 0, "the shape must use the scratch"
    cases = [_inputs(1, 3, SEG_T, gated=True, seed=51), _inputs(1, 3, SEG_T, gated=False, seed=52)]
    refs = [la.prefill_chunked(d["q"], d["k"], d["v"], alpha=d["alpha"], S0=d["S0"], z0=d["z0"]) for d in cases]
    # two calls in a row on the same stream, then one short call that needs no scratch
    outs = []
    for d in cases:
        y, S, z = _outputs(d)
        outs.append(la.prefill_chunked_noalloc(d["q"], d["k"], d["v"], y, S, z, alpha=d["alpha"], S0=d["S0"],
                                               z0=d["z0"]))
    short = _inputs(2, 2, 300, gated=True, seed=53)
    assert la.prefill_workspace_bytes(2, 2, 300, 128, 128) == 0
    ref_short = la.prefill_chunked(short["q"], short["k"], short["v"], alpha=short["alpha"], S0=short["S0"],
                                   z0=short["z0"])
    y, S, z = _outputs(short)
    out_short = la.prefill_chunked_noalloc(short["q"], short["k"], short["v"], y, S, z, alpha=short["alpha"],
                                           S0=short["S0"], z0=short["z0"])
    torch.cuda.synchronize()
    assert la.last_device_status() == 0
    for ref, out in zip(refs + [ref_short], outs + [out_short]):
        for a, b in zip(ref, out):
            assert torch.equal(a, b)


def test_noalloc_requires_outputs(la):
    d = _inputs(1, 1, 64, gated=False, seed=54)
    with pytest.raises(ValueError):
        la.prefill_chunked_noalloc(d["q"], d["k"], d["v"], None, None, None)
