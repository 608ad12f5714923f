"""CUDA path (through the C ABI) against the FP64 oracle, element by element, on
identical seeded inputs.  Tolerances: 2e-2 for BF16 inputs and 1e-5 for FP32
inputs, on the relative error of the whole tensor (max|gpu-ref| / max|ref|) and
on that of every row (every token of y, every feature row of S, the z vector of
every head), so that small late-sequence outputs are held to their own size.

Sources: LA = "Linear attention：把历史写进状态" (hs-black.github.io/posts/linear-attention);
LC = "45. Linear Attention and Recurrent State | 线性注意力与递推状态" (datawhalechina, ch. 45).
"""
import numpy as np
import pytest
import torch

from conftest import assert_close, to_oracle

pytestmark = pytest.mark.gpu

TOL = {torch.bfloat16: 2e-2, torch.float32: 1e-5}


@pytest.fixture(scope="module")
def la():
    from recurrent_state_02_gb300 import build
    build.build()
    import recurrent_state_02_gb300 as la_mod
    assert torch.cuda.is_available()
    return la_mod


def _oracle_prefill(oracle_mod, inp, eps=1e-6, threads=0):
    return oracle_mod.scan(to_oracle(inp["q"]), to_oracle(inp["k"]), to_oracle(inp["v"]),
                           alpha=to_oracle(inp["alpha"]), S0=to_oracle(inp["S0"]), z0=to_oracle(inp["z0"]),
                           eps=eps, threads=threads)


def _gpu_prefill(la, inp, chunk=64, eps=1e-6):
    d = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    y, S, z = la.prefill_chunked(d["q"], d["k"], d["v"], alpha=d["alpha"], S0=d["S0"], z0=d["z0"],
                                 chunk=chunk, eps=eps)
    assert la.last_device_status() == 0
    return y.float().cpu().numpy(), S.cpu().numpy(), z.cpu().numpy()


def _check(got, ref, tol, what=""):
    for name, g, r in zip(("y", "S", "z"), got, ref):
        assert_close(g, r, tol, f"{what} {name}")


def _inputs(dtype, B, H, T, r, dv, gated=False, with_state=False, seed=0, scale=1.0):
    from recurrent_state_02_gb300 import workloads as W
    w = W.Workload("test", B=B, H=H, T=T, r=r, dv=dv, dtype=dtype, gated=gated, seed=seed, scale=scale)
    return W.prefill_inputs(w, with_state=with_state)


# ---------------------------------------------------------------- state init

def test_state_init(la):
    S = torch.randn(3, 5, 17, 9, device="cuda")
    z = torch.randn(3, 5, 17, device="cuda")
    la.state_init(3, 5, 17, 9, S=S, z=z)
    torch.cuda.synchronize()
    assert not S.any() and not z.any()


def test_state_init_unaligned(la):
    """S and z that start 4 and 12 bytes past a 16-byte boundary, with lengths that
    are not multiples of 4: the single-float head and tail around the 16-byte
    stores, and nothing outside the arrays touched."""
    B, H, r, dv = 2, 3, 7, 5
    nS, nz = B * H * r * dv, B * H * r
    bufS = torch.randn(nS + 8, device="cuda")
    bufz = torch.randn(nz + 8, device="cuda")
    S = bufS[1:1 + nS].view(B, H, r, dv)
    z = bufz[3:3 + nz].view(B, H, r)
    before_S, before_z = bufS.clone(), bufz.clone()
    la.state_init(B, H, r, dv, S=S, z=z)
    torch.cuda.synchronize()
    assert not S.any() and not z.any()
    assert torch.equal(bufS[:1], before_S[:1]) and torch.equal(bufS[1 + nS:], before_S[1 + nS:])
    assert torch.equal(bufz[:3], before_z[:3]) and torch.equal(bufz[3 + nz:], before_z[3 + nz:])


# ------------------------------------------------------------- FP32 prefill

def test_tiny_workload_fp32(la, oracle_mod):
    """The tiny FP64 workload: FP32-rounded inputs on both sides, tolerance 1e-5."""
    from recurrent_state_02_gb300 import workloads as W
    inp = W.prefill_inputs(W.TINY)
    _check(_gpu_prefill(la, inp), _oracle_prefill(oracle_mod, inp), 1e-5, "tiny")


@pytest.mark.parametrize("gated", [False, True])
@pytest.mark.parametrize("with_state", [False, True])
def test_prefill_fp32_ragged(la, oracle_mod, gated, with_state):
    inp = _inputs(torch.float32, 2, 3, 197, 48, 24, gated=gated, with_state=with_state, seed=11)
    _check(_gpu_prefill(la, inp), _oracle_prefill(oracle_mod, inp), 1e-5, "fp32")


@pytest.mark.parametrize("r,dv", [(256, 256), (200, 160), (256, 33), (1, 129)])
def test_prefill_fp32_wide(la, oracle_mod, r, dv):
    """Widths up to 256: value columns beyond 128 go to a second CTA of the head."""
    inp = _inputs(torch.float32, 1, 2, 45, r, dv, gated=True, with_state=True, seed=12 + r + dv, scale=0.5)
    _check(_gpu_prefill(la, inp), _oracle_prefill(oracle_mod, inp), 1e-5, f"fp32 r={r} dv={dv}")


def test_prefill_fp32_wide_in_place(la, oracle_mod):
    """S0, z0 aliasing S_out, z_out with two column slices per head: no slice writes z
    before the other has read it."""
    inp = _inputs(torch.float32, 2, 2, 30, 256, 256, gated=True, with_state=True, seed=13, scale=0.5)
    ref = _oracle_prefill(oracle_mod, inp)
    d = {k: v.cuda() for k, v in inp.items()}
    S, z = d["S0"], d["z0"]
    y, _, _ = la.prefill_chunked(d["q"], d["k"], d["v"], alpha=d["alpha"], S0=S, z0=z, S_out=S, z_out=z)
    assert la.last_device_status() == 0
    _check((y.cpu().numpy(), S.cpu().numpy(), z.cpu().numpy()), ref, 1e-5, "fp32 wide in place")


# ------------------------------------------------------------- BF16 prefill

@pytest.mark.parametrize("T", [1, 17, 63, 64, 65, 5 * 64 + 17])
@pytest.mark.parametrize("dv", [64, 128])
def test_prefill_bf16_lengths(la, oracle_mod, T, dv):
    inp = _inputs(torch.bfloat16, 1, 3, T, 128, dv, seed=T + dv)
    _check(_gpu_prefill(la, inp), _oracle_prefill(oracle_mod, inp), 2e-2, f"T={T} dv={dv}")


@pytest.mark.parametrize("gated", [False, True])
@pytest.mark.parametrize("with_state", [False, True])
def test_prefill_bf16_several_tiles(la, oracle_mod, gated, with_state):
    inp = _inputs(torch.bfloat16, 2, 3, 9 * 64 + 5, 128, 128, gated=gated, with_state=with_state, seed=5)
    _check(_gpu_prefill(la, inp), _oracle_prefill(oracle_mod, inp), 2e-2, "bf16")


@pytest.mark.parametrize("chunk", [1, 32, 100])
def test_prefill_bf16_chunk_argument(la, oracle_mod, chunk):
    """Any chunk length is accepted: the result does not depend on it (LA "动手实验"),
    and the tensor-core kernel computes in chunks of 64 tokens whatever is asked for."""
    inp = _inputs(torch.bfloat16, 1, 2, 3 * 64 + 9, 128, 128, gated=True, seed=41)
    got = _gpu_prefill(la, inp, chunk=chunk)
    base = _gpu_prefill(la, inp, chunk=64)
    for g, b in zip(got, base):
        np.testing.assert_array_equal(g, b)
    _check(got, _oracle_prefill(oracle_mod, inp), 2e-2, f"chunk={chunk}")


def test_prefill_bf16_zero_gates(la, oracle_mod):
    """alpha = 0 forgets everything before it, also inside a chunk (LA '加一个门')."""
    inp = _inputs(torch.bfloat16, 1, 2, 300, 128, 128, gated=True, with_state=True, seed=8)
    inp["alpha"][0, 0, [0, 70, 127, 128, 200]] = 0.0
    inp["alpha"][0, 1, 64:128] = 0.0
    _check(_gpu_prefill(la, inp), _oracle_prefill(oracle_mod, inp), 2e-2, "zero gates")


@pytest.mark.parametrize("with_state", [False, True])
def test_prefill_bf16_tiny_gates(la, oracle_mod, with_state):
    """Chunks whose gates decay by more than e^-44 inside the chunk (alpha = 0.2 over a
    whole chunk; one alpha = 1e-20) next to ordinary ones: the kernel applies the
    gate products explicitly there instead of as row weights on V (LA '加一个门')."""
    inp = _inputs(torch.bfloat16, 1, 2, 6 * 64 + 9, 128, 128, gated=True, with_state=with_state, seed=44)
    inp["alpha"][0, 0, 64:128] = 0.2
    inp["alpha"][0, 1, 3 * 64 + 17] = 1e-20
    inp["alpha"][0, 1, 5 * 64:5 * 64 + 9] = 0.05
    _check(_gpu_prefill(la, inp), _oracle_prefill(oracle_mod, inp), 2e-2, "tiny gates")


def test_prefill_in_place_state(la, oracle_mod):
    """S0 may alias S_out and z0 may alias z_out (continuation in place)."""
    inp = _inputs(torch.bfloat16, 2, 4, 200, 128, 128, gated=True, with_state=True, seed=9)
    ref = _oracle_prefill(oracle_mod, inp)
    d = {k: v.cuda() for k, v in inp.items()}
    S, z = d["S0"], d["z0"]
    y, S_out, z_out = la.prefill_chunked(d["q"], d["k"], d["v"], alpha=d["alpha"], S0=S, z0=z, S_out=S, z_out=z)
    assert S_out.data_ptr() == S.data_ptr()
    assert la.last_device_status() == 0
    _check((y.float().cpu().numpy(), S.cpu().numpy(), z.cpu().numpy()), ref, 2e-2, "in place")


def test_prefix_causality_gpu(la):
    """LC test_prefix_causality: changing the keys and values of later tokens leaves
    earlier outputs unchanged -- here bit-identical, gated and ungated."""
    for gated in (False, True):
        inp = _inputs(torch.bfloat16, 1, 2, 200, 128, 128, gated=gated, seed=3)
        y0, _, _ = _gpu_prefill(la, inp)
        for t in (199, 150, 128, 64, 10):
            mod = {k: (v.clone() if v is not None else None) for k, v in inp.items()}
            mod["k"][:, :, t:] += 3.0
            mod["v"][:, :, t:] -= 2.0
            y1, _, _ = _gpu_prefill(la, mod)
            np.testing.assert_array_equal(y0[:, :, :t], y1[:, :, :t])


def test_prefix_causality_gates_gpu(la, oracle_mod):
    """Changing later gates leaves earlier outputs unchanged: bit-identical before the
    chunk of the first changed token; inside that chunk a chunk whose gates allow it
    carries them as row weights w_j = prod of the chunk's later gates (exact in real
    arithmetic), so earlier rows there may differ by rounding only and stay within
    the parity bar of the oracle (which is exactly causal)."""
    inp = _inputs(torch.bfloat16, 1, 2, 200, 128, 128, gated=True, seed=3)
    y0, _, _ = _gpu_prefill(la, inp)
    for t in (199, 150, 128, 64, 10):
        mod = {k: (v.clone() if v is not None else None) for k, v in inp.items()}
        mod["alpha"][:, :, t:] = 0.5
        y1, _, _ = _gpu_prefill(la, mod)
        c0 = (t // 64) * 64
        np.testing.assert_array_equal(y0[:, :, :c0], y1[:, :, :c0])
        if t > c0:
            ref, _, _ = _oracle_prefill(oracle_mod, mod)
            assert_close(y1[:, :, c0:t], ref[:, :, c0:t], 2e-2, f"gates changed from {t}")


def test_continuation_prefill_and_decode(la, oracle_mod):
    """The state is the checkpoint: prefill T1, prefill T2 from it, then decode n
    tokens one by one equals the oracle run over all T1 + T2 + n tokens."""
    from recurrent_state_02_gb300 import workloads as W
    T1, T2, n = 130, 70, 5
    inp = _inputs(torch.bfloat16, 2, 3, T1 + T2 + n, 128, 128, gated=True, seed=21)
    ref_y, ref_S, ref_z = _oracle_prefill(oracle_mod, inp)
    d = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    y1, S, z = la.prefill_chunked(d["q"][:, :, :T1].contiguous(), d["k"][:, :, :T1].contiguous(),
                                  d["v"][:, :, :T1].contiguous(), alpha=d["alpha"][:, :, :T1].contiguous())
    sl = slice(T1, T1 + T2)
    y2, S, z = la.prefill_chunked(d["q"][:, :, sl].contiguous(), d["k"][:, :, sl].contiguous(),
                                  d["v"][:, :, sl].contiguous(), alpha=d["alpha"][:, :, sl].contiguous(),
                                  S0=S, z0=z, S_out=S, z_out=z)
    ys = [y1, y2]
    for t in range(T1 + T2, T1 + T2 + n):
        ys.append(la.decode_step(d["q"][:, :, t:t + 1].contiguous(), d["k"][:, :, t:t + 1].contiguous(),
                                 d["v"][:, :, t:t + 1].contiguous(), S, z, alpha=d["alpha"][:, :, t].contiguous()))
    assert la.last_device_status() == 0
    y = torch.cat(ys, dim=2).float().cpu().numpy()
    _check((y, S.cpu().numpy(), z.cpu().numpy()), (ref_y, ref_S, ref_z), 2e-2, "continuation")


# ------------------------------------------------------------------- decode

@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("gated", [False, True])
@pytest.mark.parametrize("rdv", [(128, 128), (64, 32), (200, 256), (7, 3)])
def test_decode_step(la, oracle_mod, dtype, gated, rdv):
    from recurrent_state_02_gb300 import workloads as W
    r, dv = rdv
    w = W.DECODE.with_(B=5, H=3, r=r, dv=dv, dtype=dtype, gated=gated)
    inp = W.decode_inputs(w)
    alpha = inp["alpha"][..., None] if gated else None
    ref_y, ref_S, ref_z = oracle_mod.scan(to_oracle(inp["q"]), to_oracle(inp["k"]), to_oracle(inp["v"]),
                                          alpha=to_oracle(alpha), S0=to_oracle(inp["S"]), z0=to_oracle(inp["z"]))
    d = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    y = la.decode_step(d["q"], d["k"], d["v"], d["S"], d["z"], alpha=d["alpha"])
    assert la.last_device_status() == 0
    _check((y.float().cpu().numpy(), d["S"].cpu().numpy(), d["z"].cpu().numpy()), (ref_y, ref_S, ref_z),
           TOL[dtype], "decode")


# -------------------------------------------------------------- diagnostics

def test_wait_timeout_is_reported(la):
    """A barrier wait that runs out records LA_ERR_TIMEOUT; the context stays usable."""
    from recurrent_state_02_gb300 import _native
    assert la.last_device_status() == 0
    st = _native.lib().la_debug_wait_probe(2_000_000, torch.cuda.current_stream().cuda_stream)
    assert st == 0
    assert la.last_device_status() == _native.LA_ERR_TIMEOUT
    assert la.last_device_status() == 0
    S, z = la.state_init(2, 2, 4, 4)
    torch.cuda.synchronize()
    assert not S.any()


# ------------------------------------------------------ segmented prefill
# Few heads and a long sequence leave most SMs idle; the kernel then splits each
# sequence into segments that start from scanned states (LA "门控递推为什么能做并行
# scan？": the per-token updates are affine maps of the state and compose).

SEG_T = 47 * 64 - 21   # 47 chunks, ragged last chunk


def _segments(la, B, H, T, dv=128):
    return la.prefill_workspace_bytes(B, H, T, 128, dv)


@pytest.mark.parametrize("gated", [False, True])
@pytest.mark.parametrize("with_state", [False, True])
def test_prefill_segmented(la, oracle_mod, gated, with_state):
    assert _segments(la, 1, 3, SEG_T) > 0
    inp = _inputs(torch.bfloat16, 1, 3, SEG_T, 128, 128, gated=gated, with_state=with_state, seed=31)
    _check(_gpu_prefill(la, inp), _oracle_prefill(oracle_mod, inp), 2e-2, "segmented")


def test_prefill_segmented_dv64(la, oracle_mod):
    assert _segments(la, 2, 1, SEG_T, dv=64) > 0
    inp = _inputs(torch.bfloat16, 2, 1, SEG_T, 128, 64, gated=True, with_state=True, seed=32)
    _check(_gpu_prefill(la, inp), _oracle_prefill(oracle_mod, inp), 2e-2, "segmented dv64")


def test_prefill_segmented_zero_gates(la, oracle_mod):
    """alpha = 0 at and around segment and part boundaries is exact: nothing before it survives."""
    assert _segments(la, 1, 2, SEG_T) > 0
    inp = _inputs(torch.bfloat16, 1, 2, SEG_T, 128, 128, gated=True, with_state=True, seed=33)
    for t in (0, 63, 64, 65, 1535, 1536, 1537, 2000, SEG_T - 1):
        inp["alpha"][0, 0, t] = 0.0
    inp["alpha"][0, 1, 1500:1600] = 0.0
    _check(_gpu_prefill(la, inp), _oracle_prefill(oracle_mod, inp), 2e-2, "segmented zero gates")


def test_prefill_segmented_in_place(la, oracle_mod):
    """S0 may alias S_out with segments: every segment reads its start state from the workspace."""
    assert _segments(la, 1, 3, SEG_T) > 0
    inp = _inputs(torch.bfloat16, 1, 3, SEG_T, 128, 128, gated=True, with_state=True, seed=34)
    ref = _oracle_prefill(oracle_mod, inp)
    d = {k: v.cuda() for k, v in inp.items()}
    S, z = d["S0"], d["z0"]
    y, _, _ = la.prefill_chunked(d["q"], d["k"], d["v"], alpha=d["alpha"], S0=S, z0=z, S_out=S, z_out=z)
    assert la.last_device_status() == 0
    _check((y.float().cpu().numpy(), S.cpu().numpy(), z.cpu().numpy()), ref, 2e-2, "segmented in place")


def test_prefill_workspace_errors(la):
    """A segmenting shape without (enough, aligned) workspace is refused before any launch."""
    from recurrent_state_02_gb300 import _native
    need = _segments(la, 1, 3, SEG_T)
    assert need > 0
    inp = _inputs(torch.bfloat16, 1, 3, SEG_T, 128, 128, seed=35)
    d = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    y = torch.empty_like(d["v"])
    S = torch.empty(1, 3, 128, 128, device="cuda")
    z = torch.empty(1, 3, 128, device="cuda")
    ws = torch.empty(need + 512, device="cuda", dtype=torch.uint8)
    L = _native.lib()
    P = lambda t: t.data_ptr()
    sh = torch.cuda.current_stream().cuda_stream

    def call(wptr, wbytes):
        return L.la_prefill_chunked(P(d["q"]), P(d["k"]), P(d["v"]), _native.LA_DTYPE_BF16, None, None, None,
                                    1, 3, SEG_T, 128, 128, 64, 1e-6, P(y), P(S), P(z), wptr, wbytes, sh)

    assert call(None, 0) == _native.LA_ERR_WORKSPACE
    assert call(P(ws), need - 1) == _native.LA_ERR_WORKSPACE
    assert call(P(ws) + 16, need) == _native.LA_ERR_ALIGN
    assert call(P(ws), need) == 0
    torch.cuda.synchronize()
    assert la.last_device_status() == 0


# ------------------------------------------------------- packed sequences
# Sequences of different lengths packed one after another (token-major
# [total, H, d]), each from its own state: every sequence must equal the oracle
# run over that sequence alone.

VARLEN_LENS = [0, 1, 63, 64, 65, 300, 17]


def _varlen_inputs(gated, seed):
    from recurrent_state_02_gb300 import workloads as W
    lens = VARLEN_LENS
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    H = 2
    base = W.prefill_inputs(W.Workload("varlen", B=1, H=H, T=int(cu[-1]), dtype=torch.bfloat16, gated=gated,
                                       seed=seed))
    g = torch.Generator().manual_seed(seed + 1)
    B = len(lens)
    S0 = (torch.randn(B, H, 128, 128, generator=g) * 0.1).float()
    z0 = (torch.rand(B, H, 128, generator=g) * 10 + 1).float()
    return base, cu, S0, z0


@pytest.mark.parametrize("gated", [False, True])
def test_prefill_varlen(la, oracle_mod, gated):
    base, cu, S0, z0 = _varlen_inputs(gated, 61)
    pack = lambda x: x[0].permute(1, 0, 2).contiguous().cuda()          # [1,H,T,d] -> [T,H,d]
    alpha = base["alpha"][0].permute(1, 0).contiguous().cuda() if gated else None
    y, S, z = la.prefill_varlen(pack(base["q"]), pack(base["k"]), pack(base["v"]), torch.from_numpy(cu).cuda(),
                                alpha=alpha, S0=S0.cuda(), z0=z0.cuda())
    assert la.last_device_status() == 0
    y, S, z = y.float().cpu(), S.cpu(), z.cpu()
    for b in range(len(VARLEN_LENS)):
        lo, hi = int(cu[b]), int(cu[b + 1])
        if hi == lo:   # an empty sequence hands its state on unchanged
            assert torch.equal(S[b], S0[b]) and torch.equal(z[b], z0[b])
            continue
        sl = lambda x: x[:, :, lo:hi].contiguous()
        ref = oracle_mod.scan(to_oracle(sl(base["q"])), to_oracle(sl(base["k"])), to_oracle(sl(base["v"])),
                              alpha=to_oracle(base["alpha"][:, :, lo:hi].contiguous()) if gated else None,
                              S0=to_oracle(S0[b:b + 1]), z0=to_oracle(z0[b:b + 1]), eps=1e-6)
        got = (y[lo:hi].permute(1, 0, 2)[None].numpy(), S[b:b + 1].numpy(), z[b:b + 1].numpy())
        _check(got, ref, 2e-2, f"varlen seq {b} (T={hi - lo})")


def test_prefill_varlen_bad_lengths(la, oracle_mod):
    """Offsets that run backwards are refused on the device: that sequence is
    skipped, the error is recorded, and the other sequences are still exact."""
    base, cu, S0, z0 = _varlen_inputs(False, 62)
    bad = cu.copy()
    bad[3] = bad[2] - 1   # sequence 2 would have negative length
    pack = lambda x: x[0].permute(1, 0, 2).contiguous().cuda()
    y, S, z = la.prefill_varlen(pack(base["q"]), pack(base["k"]), pack(base["v"]), torch.from_numpy(bad).cuda(),
                                S0=S0.cuda(), z0=z0.cuda())
    from recurrent_state_02_gb300 import _native
    assert la.last_device_status() == _native.LA_ERR_SHAPE
    assert la.last_device_status() == 0
    lo, hi = int(bad[5]), int(bad[6])   # a well-formed sequence
    sl = lambda x: x[:, :, lo:hi].contiguous()
    ref = oracle_mod.scan(to_oracle(sl(base["q"])), to_oracle(sl(base["k"])), to_oracle(sl(base["v"])),
                          S0=to_oracle(S0[5:6]), z0=to_oracle(z0[5:6]), eps=1e-6)
    got = (y.float().cpu()[lo:hi].permute(1, 0, 2)[None].numpy(), S.cpu()[5:6].numpy(), z.cpu()[5:6].numpy())
    _check(got, ref, 2e-2, "varlen next to a bad sequence")


# ------------------------------------------------------ short continuations
# A BF16 call of at most 32 tokens at r = dv = 128 takes the decode-shaped token
# walk (the state stays in registers for the whole run; FP32 arithmetic; the
# tokens are staged in halves of 16).
SHORT_CASES = [
    # B, H, T, gated, with_state
    (3, 5, 1, False, True),
    (2, 3, 2, True, True),
    (4, 2, 7, True, False),
    (2, 4, 16, False, False),
    (1, 6, 16, True, True),
    (2, 3, 17, True, True),     # one token into the second half
    (3, 2, 24, False, True),
    (2, 2, 32, True, False),    # the most the walk takes
    (1, 3, 32, False, True),
    (2, 2, 33, True, True),     # one more: the chunk kernel
]


@pytest.mark.parametrize("B,H,T,gated,with_state", SHORT_CASES,
                         ids=[f"B{c[0]}H{c[1]}T{c[2]}-g{int(c[3])}-s{int(c[4])}" for c in SHORT_CASES])
def test_prefill_short_continuation(la, oracle_mod, B, H, T, gated, with_state):
    inp = _inputs(torch.bfloat16, B, H, T, 128, 128, gated=gated, with_state=with_state, seed=600 + T)
    _check(_gpu_prefill(la, inp), _oracle_prefill(oracle_mod, inp), 2e-2, f"short T={T}")


@pytest.mark.parametrize("T,gated", [(8, False), (32, True)])
def test_prefill_short_continuation_unaligned_state(la, oracle_mod, T, gated):
    """A carried S0 that is 4-byte aligned only: the call takes the chunk kernel
    instead of the token walk (which reads S0 as float4) and still matches."""
    inp = _inputs(torch.bfloat16, 2, 3, T, 128, 128, gated=gated, with_state=True, seed=640 + T)
    d = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    n = d["S0"].numel()
    buf = torch.empty(n + 4, device="cuda", dtype=torch.float32)
    S0 = buf[1:1 + n].view_as(d["S0"])
    S0.copy_(d["S0"])
    y, S, z = la.prefill_chunked(d["q"], d["k"], d["v"], alpha=d["alpha"], S0=S0, z0=d["z0"])
    assert la.last_device_status() == 0
    _check((y.float().cpu().numpy(), S.cpu().numpy(), z.cpu().numpy()), _oracle_prefill(oracle_mod, inp), 2e-2,
           f"short T={T} from a 4-byte aligned state")


def test_prefill_short_continuation_in_place_chain(la, oracle_mod):
    """Prefill 100 tokens, then continuations of 1, 5, 16 and 29 tokens in place
    (S0 = S_out), against one oracle pass over all 151 tokens."""
    inp = _inputs(torch.bfloat16, 2, 3, 151, 128, 128, gated=True, with_state=True, seed=77)
    ref = _oracle_prefill(oracle_mod, inp)
    d = {k: (v.cuda() if v is not None else None) for k, v in inp.items()}
    S, z = d["S0"].clone(), d["z0"].clone()
    ys = []
    for a, b in ((0, 100), (100, 101), (101, 106), (106, 122), (122, 151)):
        part = {n: (d[n][:, :, a:b].contiguous() if d[n] is not None else None) for n in ("q", "k", "v", "alpha")}
        y, _, _ = la.prefill_chunked(part["q"], part["k"], part["v"], alpha=part["alpha"], S0=S, z0=z,
                                     S_out=S, z_out=z)
        ys.append(y)
    assert la.last_device_status() == 0
    got = (torch.cat(ys, dim=2).float().cpu().numpy(), S.cpu().numpy(), z.cpu().numpy())
    _check(got, ref, 2e-2, "prefill then short continuations")
