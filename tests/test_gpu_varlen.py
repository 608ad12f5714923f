"""Packed sequences split into segments: la_prefill_varlen on batches where some
sequences are long enough for the plan kernel to cut them into segments (a state
pass and a scan give each segment its start state: "门控递推为什么能做并行 scan？" of
[LA], a run of tokens is one affine map of the state).

Every sequence is held to the oracle run over that sequence alone, from its own
S0, z0 (BF16 bar 2e-2, as the other prefill tests).  The plan's segment length
and the segment count of each sequence are read back from the head of the
workspace (the length at byte 0, the per-sequence int4 records from byte 256:
segments, first start-state slot, first boundary; the item table of (sequence,
segment) pairs after them, from the next 256-byte boundary), so each test also
checks that the split it is about took place and that the chunk kernel's CTAs
start with the longest segments.  Sequences of at most 32 tokens (empty ones
included) take the token walk instead: no segment, no item.
"""
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
    assert torch.cuda.is_available()
    return la_mod


def _packed(lens, H, dv, gated, seed, zero_gates=()):
    """q, k, v [total, H, d] BF16 and alpha [total, H] FP32 (token-major), cu_seqlens,
    S0 [B, H, 128, dv] ~ N(0, 0.01), z0 [B, H, 128] ~ U(1, 11).  zero_gates: absolute
    token rows whose gate is set to 0 (every head)."""
    from recurrent_state_02_gb300 import workloads as W
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    total = int(cu[-1])
    base = W.prefill_inputs(W.Workload("varlen", B=1, H=H, T=total, dv=dv, dtype=torch.bfloat16, gated=gated,
                                       seed=seed))
    tok = lambda x: x[0].permute(1, 0, 2).contiguous()
    alpha = base["alpha"][0].permute(1, 0).contiguous() if gated else None
    if alpha is not None:
        for t in zero_gates:
            alpha[t] = 0.0
    g = torch.Generator().manual_seed(seed + 1)
    B = len(lens)
    S0 = (torch.randn(B, H, 128, dv, generator=g) * 0.1).float()
    z0 = (torch.rand(B, H, 128, generator=g) * 10 + 1).float()
    return dict(q=tok(base["q"]), k=tok(base["k"]), v=tok(base["v"]), alpha=alpha, cu=cu, S0=S0, z0=z0)


def _run(la, d, in_place=False):
    B = len(d["cu"]) - 1
    total, H, _ = d["q"].shape
    dv = d["v"].shape[2]
    need = la.varlen_workspace_bytes(B, H, total, 128, dv)
    ws = torch.zeros(max(need, 256), device="cuda", dtype=torch.uint8)
    g = {n: (d[n].cuda() if d[n] is not None else None) for n in ("q", "k", "v", "alpha", "S0", "z0")}
    kw = dict(S_out=g["S0"], z_out=g["z0"]) if in_place else {}
    y, S, z = la.prefill_varlen(g["q"], g["k"], g["v"], torch.from_numpy(d["cu"]).cuda(), alpha=g["alpha"],
                                S0=g["S0"], z0=g["z0"], workspace=ws if need else None, **kw)
    status = la.last_device_status()
    plan = None
    if need:
        w = ws.cpu()
        L = int(w[:4].view(torch.int32)[0])
        info = w[256:256 + 16 * B].view(torch.int32).view(B, 4).numpy()
        off = 256 + (16 * B + 255) // 256 * 256
        n_items = int(np.sum(info[:, 0]))
        items = w[off:off + 8 * n_items].view(torch.int32).view(n_items, 2).numpy()
        plan = (L, info, items, dv)
    return (y.float().cpu(), S.cpu(), z.cpu()), status, plan


def _order_key(c):
    """Larger items first: c itself below 64, then 8 buckets per octave."""
    if c < 64:
        return -c
    o = c.bit_length() - 1
    return -(64 + 8 * (o - 6) + ((c >> (o - 3)) & 7))


WALK_MAX = 32   # a valid sequence of at most this many tokens takes the token walk (dv = 128)


def _check_plan(plan, lens, expect_split=True, invalid=()):
    assert plan is not None, "no workspace: the plan does not segment at these sizes"
    L, info, items, dv = plan
    walk_max = WALK_MAX if dv == 128 else -1
    assert L >= 16
    # a sequence with bad bounds counts as empty; a short valid one takes no segment
    chunks = [0 if b in invalid else (n + 63) // 64 for b, n in enumerate(lens)]
    walked = [b not in invalid and n <= walk_max for b, n in enumerate(lens)]
    want = [0 if walked[b] else (c + L - 1) // L if (expect_split and c > L) else 1 for b, c in enumerate(chunks)]
    assert list(info[:, 0]) == want, (L, list(info[:, 0]), want)
    if expect_split:
        assert max(want) > 1, "no sequence was split"
        # boundaries and start-state slots are numbered in sequence order
        bd = np.concatenate([[0], np.cumsum([max(0, n - 1) for n in want])])[:-1]
        assert list(info[:, 2]) == list(bd)
        slots = np.concatenate([[0], np.cumsum([n if n > 1 else 0 for n in want])])[:-1]
        assert [int(info[b, 1]) for b in range(len(lens)) if want[b] > 1] == \
            [int(slots[b]) for b in range(len(lens)) if want[b] > 1]
    # every segment once, longest first
    pairs = sorted(map(tuple, items.tolist()))
    assert pairs == sorted((b, g) for b in range(len(lens)) for g in range(want[b]))
    seg_chunks = lambda b, g: L if g + 1 < want[b] else chunks[b] - (want[b] - 1) * L
    keys = [_order_key(seg_chunks(b, g)) for b, g in items.tolist()]
    assert keys == sorted(keys)
    return L


def _check_seqs(oracle_mod, d, got, skip=()):
    y, S, z = got
    cu = d["cu"]
    for b in range(len(cu) - 1):
        if b in skip:
            continue
        lo, hi = int(cu[b]), int(cu[b + 1])
        if hi == lo:   # an empty sequence hands its state on unchanged
            assert torch.equal(S[b], d["S0"][b]) and torch.equal(z[b], d["z0"][b])
            continue
        sl = lambda x: x[lo:hi].permute(1, 0, 2)[None].contiguous()
        ref = oracle_mod.scan(to_oracle(sl(d["q"])), to_oracle(sl(d["k"])), to_oracle(sl(d["v"])),
                              alpha=to_oracle(d["alpha"][lo:hi].permute(1, 0)[None].contiguous())
                              if d["alpha"] is not None else None,
                              S0=to_oracle(d["S0"][b:b + 1]), z0=to_oracle(d["z0"][b:b + 1]), eps=1e-6)
        g = (y[lo:hi].permute(1, 0, 2)[None].numpy(), S[b:b + 1].numpy(), z[b:b + 1].numpy())
        for name, a, r in zip(("y", "S", "z"), g, ref):
            assert_close(a, r, 2e-2, f"varlen seq {b} (T={hi - lo}) {name}")


# long sequences among short and empty ones; the long ones span several 16-chunk
# segments, with ragged ends
MIXED = [5000, 0, 100, 2100, 64, 1, 3000, 17]


@pytest.mark.parametrize("gated", [False, True])
def test_varlen_segments_mixed(la, oracle_mod, gated):
    d = _packed(MIXED, 2, 128, gated, seed=70 + gated)
    got, status, plan = _run(la, d)
    assert status == 0
    _check_plan(plan, MIXED)
    _check_seqs(oracle_mod, d, got)


def test_varlen_segments_zero_gates(la, oracle_mod):
    """Zero gates inside the long sequences: on the first token of a segment, on the
    last one, and mid-segment; the maps of the parts before them must vanish."""
    lens = [4200, 33, 2500]
    d = _packed(lens, 2, 128, True, seed=73,
                zero_gates=(1024, 2047, 3000, 4200 + 33 + 1500))
    got, status, plan = _run(la, d)
    assert status == 0
    _check_plan(plan, lens)
    _check_seqs(oracle_mod, d, got)


def test_varlen_segments_in_place(la, oracle_mod):
    """S0 and z0 are also S_out and z_out: the first segment of a split sequence must
    not read a state that its last segment has already written."""
    lens = [3100, 70, 0, 2600]
    d = _packed(lens, 3, 128, True, seed=74)
    got, status, plan = _run(la, d, in_place=True)
    assert status == 0
    _check_plan(plan, lens)
    _check_seqs(oracle_mod, d, got)


def test_varlen_segments_dv64(la, oracle_mod):
    lens = [2900, 5, 1200, 640]
    d = _packed(lens, 2, 64, True, seed=75)
    got, status, plan = _run(la, d)
    assert status == 0
    _check_plan(plan, lens)
    _check_seqs(oracle_mod, d, got)


def test_varlen_segments_many_sequences(la, oracle_mod):
    """More sequences than the plan kernel's 1024 threads: its prefix sums carry
    across tiles.  Three long sequences, one in each tile and one at the end."""
    rng = np.random.default_rng(76)
    lens = [int(x) for x in rng.integers(0, 40, 1500)]
    for i in (5, 1100, 1499):
        lens[i] = 2300
    d = _packed(lens, 1, 128, False, seed=76)
    got, status, plan = _run(la, d)
    assert status == 0
    _check_plan(plan, lens)
    _check_seqs(oracle_mod, d, got)


def test_varlen_bad_lengths_disable_segments(la, oracle_mod):
    """The last sequence runs past the total: nothing is split, the error is
    recorded, and the other sequences (long ones included) are still exact."""
    lens = [3000, 100, 2000, 500]
    d = _packed(lens, 2, 128, False, seed=77)
    d["cu"] = d["cu"].copy()
    d["cu"][-1] += 5
    got, status, plan = _run(la, d)
    from recurrent_state_02_gb300 import _native
    assert status == _native.LA_ERR_SHAPE
    assert la.last_device_status() == 0
    _check_plan(plan, lens, expect_split=False, invalid=(3,))
    _check_seqs(oracle_mod, d, got, skip=(3,))


def test_varlen_segments_exact_and_single_token_tails(la, oracle_mod):
    """Every sequence split: one ends exactly on a segment boundary (2048 tokens,
    two segments of 16 chunks), one leaves a last segment of a single token, and
    one a last segment of a single chunk."""
    lens = [2048, 2049, 1088, 3000]
    d = _packed(lens, 2, 128, True, seed=78)
    got, status, plan = _run(la, d)
    assert status == 0
    L = _check_plan(plan, lens)
    assert L == 16   # a batch this small keeps the minimum segment length
    _check_seqs(oracle_mod, d, got)


def test_varlen_segments_beyond_the_plan_cache(la, oracle_mod):
    """5000 sequences: the plan keeps the chunk counts of the first 4096 in shared
    memory and reads the others again; long sequences on both sides of that mark."""
    rng = np.random.default_rng(79)
    lens = [int(x) for x in rng.integers(0, 12, 5000)]
    for i in (100, 4095, 4096, 4999):
        lens[i] = 2200
    d = _packed(lens, 1, 128, False, seed=79)
    got, status, plan = _run(la, d)
    assert status == 0
    _check_plan(plan, lens)
    _check_seqs(oracle_mod, d, got)


def _ragged_short_lens(seed):
    rng = np.random.default_rng(seed)
    lens = [int(x) for x in rng.integers(0, 33, 300)]   # 0 .. 32 tokens, empty ones included
    lens[7], lens[150] = 1500, 33                        # a long prompt, and one token past the walk
    return lens


def test_varlen_ragged_short_continuations(la, oracle_mod):
    """300 requests of 0 to 32 new tokens each from its own state, gated, in place
    (the token walk), beside one long prompt and one of 33 tokens (the chunk kernel);
    a few gates are exactly 0 (a reset inside a request)."""
    lens = _ragged_short_lens(80)
    cu = np.concatenate([[0], np.cumsum(lens)])
    zeros = [int(cu[b]) + lens[b] // 2 for b in (3, 40, 200) if lens[b] > 0] + [int(cu[7]) + 700]
    d = _packed(lens, 2, 128, True, seed=80, zero_gates=zeros)
    got, status, plan = _run(la, d, in_place=True)
    assert status == 0
    _check_plan(plan, lens)
    _check_seqs(oracle_mod, d, got)


def test_varlen_ragged_short_unaligned_state(la, oracle_mod):
    """The same batch with S0 only 4-byte aligned: the walk (which reads S0 as
    float4) is not used, and every sequence takes the chunk kernel."""
    lens = _ragged_short_lens(81)
    d = _packed(lens, 2, 128, False, seed=81)
    B, H = len(lens), 2
    total = int(d["cu"][-1])
    g = {n: d[n].cuda() for n in ("q", "k", "v")}
    n = d["S0"].numel()
    buf = torch.empty(n + 4, device="cuda", dtype=torch.float32)
    S0 = buf[1:1 + n].view_as(d["S0"])
    S0.copy_(d["S0"].cuda())
    y, S, z = la.prefill_varlen(g["q"], g["k"], g["v"], torch.from_numpy(d["cu"]).cuda(), S0=S0, z0=d["z0"].cuda())
    assert la.last_device_status() == 0
    assert y.shape == (total, H, 128) and S.shape == (B, H, 128, 128)
    _check_seqs(oracle_mod, d, (y.float().cpu(), S.cpu(), z.cpu()))


@pytest.mark.parametrize("in_place", [False, True])
def test_varlen_no_tokens(la, in_place):
    """A packed batch of three empty requests (no tokens at all): every state is
    handed on unchanged, bit for bit (the walk copies it), in place or not."""
    B, H = 3, 2
    g = torch.Generator().manual_seed(82)
    S0 = (torch.randn(B, H, 128, 128, generator=g) * 0.1).cuda()
    z0 = (torch.rand(B, H, 128, generator=g) * 10 + 1).cuda()
    S0c, z0c = S0.clone(), z0.clone()
    q = torch.empty(0, H, 128, device="cuda", dtype=torch.bfloat16)
    cu = torch.zeros(B + 1, device="cuda", dtype=torch.int32)
    kw = dict(S_out=S0, z_out=z0) if in_place else {}
    y, S, z = la.prefill_varlen(q, q, q, cu, S0=S0, z0=z0, **kw)
    assert la.last_device_status() == 0
    assert y.shape == (0, H, 128)
    assert torch.equal(S.cpu(), S0c.cpu()) and torch.equal(z.cpu(), z0c.cpu())

