#!/usr/bin/env python
"""Benchmark of the linear-attention hot path on GB300.

One step = the whole hot path over one batch of the ungated prefill workload
(B=4, H=16, T=4096, r=dv=128, BF16, chunk 64): la_state_init (zero S/z),
la_prefill_chunked over the batch from that state (state updated in place),
then la_decode_step of one more token per request on the resulting state.
Tokens per step = B * (T + 1).  Inputs are synthetic (seeded), resident in HBM
when timing starts, and rotated over 4 sets (> L2) so no step reads a warm L2.
Each step is replayed as a CUDA graph of its three kernel launches.

Printed (rank 0, one JSON line): tokens/s of the step, the prefill kernel's
roofline (algorithmic bytes / mean launch time vs measured HBM bandwidth), the
decode step on its own workload (B=256, H=16) in GB/s, the gated (B=2, H=16,
T=16384) and long (B=1, H=32, T=65536) prefill workloads with their own
rooflines, the delta-rule memory on the prefill's shape (against the FP32 ALU
peak), the backward pass of the gated prefill (the whole call against measured
HBM), an end-to-end figure
through the public API with host buffers, clocks sampled during timing, and
the FP64 CPU oracle timed on the host cores.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "prefill tokens/s (B4 H16 T4096 d128) & decode GB/s; % of roofline"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
PROFILES = os.path.join(ROOT, "profiles")
FALLBACK_HBM_GBS = 6800.0
N_ROT = 4


# ----------------------------------------------------------------- helpers

def prefill_bytes(B, H, T, r, dv, with_state_in=True):
    """Algorithmic bytes of one prefill launch: q, k, v read and y written
    (BF16, 2*(r+r+dv+dv) bytes per token-head = 1024 at r = dv = 128), the final
    state written and, when given, the initial state read (FP32 r*dv + r per head)."""
    per_token_head = 2 * (2 * r + 2 * dv)
    state = 4 * (r * dv + r)
    return B * H * T * per_token_head + B * H * state * (2 if with_state_in else 1)


def prefill_flops(B, H, T, r, dv, chunk=64):
    """Algorithmic FLOPs of the chunked prefill: per token and head the scores and
    the in-chunk values (2 C r + 2 C dv) and the state read and write (4 r dv)."""
    return B * H * T * (2 * chunk * r + 2 * chunk * dv + 4 * r * dv)


def decode_bytes(B, H, r, dv, elem=2):
    """S and z read and written (FP32), q, k, v read and y written (elem bytes)."""
    return B * H * (2 * 4 * (r * dv + r) + elem * (2 * r + 2 * dv))


def varlen_bytes(B, H, total_T, r, dv, elem=2):
    """A packed batch from zero states: q, k, v read and y written (elem bytes) per
    token-head, and each sequence's final S and z written (FP32)."""
    return total_T * H * elem * (2 * r + 2 * dv) + B * H * 4 * (r * dv + r)


def short_bytes(B, H, T, r, dv, gated, elem=2):
    """A short continuation from a carried state: S and z read and written once
    (FP32), and per token q, k, v read and y written (elem bytes) and the gate (FP32)."""
    return B * H * (2 * 4 * (r * dv + r) + T * (elem * (2 * r + 2 * dv) + (4 if gated else 0)))


def delta_flops(B, H, T, r, dv):
    """Algorithmic FLOPs of one delta-rule launch: per token and head, the read
    S^T k, the rank-1 write and the read S^T q, 2 r dv each."""
    return B * H * T * 6 * r * dv


def delta_bytes(B, H, T, r, dv, elem=2):
    """Compulsory HBM bytes of one delta-rule call: q, k, v read and y written
    (elem bytes each), beta read and the final state written (FP32)."""
    return B * H * (T * (elem * (2 * r + 2 * dv) + 4) + 4 * r * dv)


def backward_flops(B, H, T, r, dv, gated):
    """Algorithmic FLOPs of the backward: per token and head, the state write and
    the read S_t dn_t for dq (2 r dv each), the write of G and the reads G_t v_t
    and G_t^T k~_t for dk and dv (2 r dv each), plus the gate's scaling of S and
    G (r dv each) when gated."""
    return B * H * T * (10 + (2 if gated else 0)) * r * dv


def backward_bytes(B, H, T, r, dv, gated, elem=2):
    """Compulsory HBM bytes of one backward call without carried states: q, k, v,
    y and dy read, dq, dk and dv written (elem bytes each), alpha read and dalpha
    written (FP32, gated only), dS0 and dz0 written (FP32)."""
    per_token_head = elem * (2 * r + 2 * dv) + elem * (2 * r + dv) + (8 if gated else 0)
    return B * H * (T * per_token_head + 4 * (r * dv + r))


def fp32_alu_peak_tflops(sm_count):
    """FP32 FMA peak of the CUDA cores: SMs x 128 FP32 lanes x 2 FLOP x the
    maximum SM clock (MEASURED_PEAKS.json, else the nominal 2070 MHz)."""
    try:
        with open(PEAKS_FILE) as f:
            mhz = float(json.load(f)["sm_max_mhz"])
    except Exception:
        mhz = 2070.0
    return sm_count * 128 * 2 * mhz * 1e6 / 1e12


def read_peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def source_sha1(paths):
    """First 12 hex digits of the SHA-1 of the concatenated source files."""
    h = hashlib.sha1()
    for path in paths:
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:12]


def kernel_sources(name):
    """The files a kernel is compiled from (its .cu and the headers it includes)."""
    csrc = os.path.join(ROOT, "recurrent_state_02_gb300", "csrc")
    common = ("tc_common.cuh",) if name in ("prefill_tc.cu", "delta.cu", "delta_tc.cu") else ()
    if name == "delta_tc.cu":
        common += ("delta_tc.h",)
    return [os.path.join(csrc, f) for f in (name, "kernels.h", "sm103_ptx.cuh") + common]


def profile_traffic(kernel, workload, src):
    """DRAM bytes per launch from a committed ncu summary, only when that summary
    was taken on the current kernel source (else None)."""
    sha = source_sha1(src)
    if not os.path.isdir(PROFILES):
        return None
    for name in sorted(os.listdir(PROFILES)):
        if not name.endswith((".txt", ".md")):
            continue
        fields = {}
        for line in open(os.path.join(PROFILES, name)):
            if "=" in line and line.strip().startswith("traffic."):
                k, v = line.strip().split("=", 1)
                fields[k.strip()] = v.strip()
        if (fields.get("traffic.kernel") == kernel and fields.get("traffic.workload") == workload
                and fields.get("traffic.source_sha1") == sha):
            try:
                return float(fields["traffic.dram_bytes_per_launch"])
            except (KeyError, ValueError):
                return None
    return None


class ClockSampler:
    """nvidia-smi samples (every 100 ms) of SM clock, power and clock-event reasons."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.lines = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.gpu_index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((ts, float(parts[1]), float(parts[2]), parts[5:9], parts[4]))
            except ValueError:
                continue
        window = [r for r in rows if t0 - 0.15 <= r[0] <= t1 + 0.15] or rows
        if not window:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in window for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in window), "sm_max_mhz": max(r[2] for r in window),
                "reasons": reasons, "samples": len(window)}


def reduce_max(values, device, dist=None):
    """Max over ranks of a list of floats (timings); identity without a process group."""
    if dist is None:
        return list(values)
    import torch
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def whole_job_rate(units_per_rank_step, world, steps, seconds):
    """Units all ranks processed per second, against the slowest rank's time."""
    return units_per_rank_step * world * steps / seconds


def gpu_index(local_rank):
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [v for v in vis.split(",") if v.strip()]
        if local_rank < len(ids):
            return ids[local_rank]
    return str(local_rank)


# --------------------------------------------------------- CPU oracle legs

def oracle_tokens_per_s(w, seconds, max_tokens=None):
    """Times the FP64 oracle (token recurrence, all host cores) over all B*H heads of
    the workload, on the first T' tokens (T' <= T, sized to ~`seconds`).
    Returns (tokens/s, cores, sample description, elapsed)."""
    import numpy as np
    import torch

    import oracle
    from recurrent_state_02_gb300 import workloads as W

    oracle.build()
    cores = oracle.num_cpus()
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    # calibrate on a short prefix, then size the sample
    gates = lambda inp: None if inp["alpha"] is None else inp["alpha"].numpy()
    Tc = min(w.T, 64)
    inp = W.prefill_inputs(w.with_(T=Tc))
    t0 = time.perf_counter()
    oracle.scan(bits(inp["q"]), bits(inp["k"]), bits(inp["v"]), alpha=gates(inp), threads=cores)
    per_token = (time.perf_counter() - t0) / (w.B * Tc)
    Ts = int(max(1, min(w.T, seconds / max(per_token, 1e-9) / w.B)))
    if max_tokens:
        Ts = min(Ts, max(1, max_tokens // w.B))
    inp = W.prefill_inputs(w.with_(T=Ts))
    q, k, v, alpha = bits(inp["q"]), bits(inp["k"]), bits(inp["v"]), gates(inp)
    reps, elapsed = 0, 0.0
    while True:
        t0 = time.perf_counter()
        oracle.scan(q, k, v, alpha=alpha, eps=w.eps, threads=cores)
        elapsed += time.perf_counter() - t0
        reps += 1
        if elapsed >= seconds or reps >= 8:
            break
    tok = w.B * Ts * reps
    desc = (f"FP64 token recurrence{' with gates' if w.gated else ''} on {cores} threads over all {w.B}x{w.H} "
            f"heads of '{w.name}', first {Ts} of "
            f"{w.T} tokens, {reps} pass(es), {elapsed:.1f} s")
    return tok / elapsed, cores, desc, elapsed


def oracle_rate(kind, w, seconds):
    """Times the FP64 oracle of the delta rule (kind "delta") or of the backward
    ("backward", gated) over all B*H heads of the workload on the first T' tokens,
    T' sized to about `seconds` from a 32-token calibration.  Returns the
    cpu_baseline object (tokens/s)."""
    import numpy as np
    import torch

    import oracle
    from recurrent_state_02_gb300 import workloads as W

    oracle.build()
    cores = oracle.num_cpus()
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)

    def run(Tn):
        if kind == "delta":
            d = W.delta_inputs(w.with_(T=Tn))
            t0 = time.perf_counter()
            oracle.delta(bits(d["q"]), bits(d["k"]), bits(d["v"]), beta=d["beta"].numpy(), threads=cores)
        else:
            d = W.prefill_inputs(w.with_(T=Tn))
            dy = np.random.default_rng(0).standard_normal((w.B, w.H, Tn, w.dv))
            t0 = time.perf_counter()
            oracle.backward(bits(d["q"]), bits(d["k"]), bits(d["v"]), dy, alpha=d["alpha"].numpy(), eps=w.eps,
                            threads=cores)
        return time.perf_counter() - t0

    per_token = run(32) / (w.B * 32)
    Ts = int(max(1, min(w.T, seconds / max(per_token, 1e-9) / w.B)))
    elapsed = run(Ts)
    what = "delta-rule memory" if kind == "delta" else "gradients of the gated token recurrence"
    return {"value": w.B * Ts / elapsed, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"FP64 {what} on {cores} threads over all {w.B}x{w.H} heads of '{w.name}', first {Ts} of "
                      f"{w.T} tokens, {elapsed:.1f} s"}


def run_reference(args, rank, world):
    """Reference arm: the FP64 CPU oracle, as it stands, on the host cores."""
    if rank != 0:
        return
    from recurrent_state_02_gb300 import workloads as W
    w = W.UNGATED
    budget = 120.0
    per_step = max(0.05, budget / max(1, args.steps + args.warmup))
    # warm-up steps (untimed), then exactly K timed steps
    import numpy as np
    import torch

    import oracle
    oracle.build()
    cores = oracle.num_cpus()
    bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
    Tc = 32
    inp = W.prefill_inputs(w.with_(T=Tc))
    t0 = time.perf_counter()
    oracle.scan(bits(inp["q"]), bits(inp["k"]), bits(inp["v"]), threads=cores)
    per_token = (time.perf_counter() - t0) / (w.B * Tc)
    Ts = int(max(1, min(w.T, per_step / max(per_token, 1e-9) / w.B)))
    inp = W.prefill_inputs(w.with_(T=Ts + 1))
    q, k, v = bits(inp["q"]), bits(inp["k"]), bits(inp["v"])
    for _ in range(args.warmup):
        oracle.scan(q, k, v, eps=w.eps, threads=cores)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.scan(q, k, v, eps=w.eps, threads=cores)
    el = time.perf_counter() - t0
    tokens = w.B * (Ts + 1) * args.steps
    value = tokens / el
    sample = (f"each step: FP64 token recurrence over all {w.B}x{w.H} heads of '{w.name}', first {Ts + 1} of "
              f"{w.T + 1} tokens (prefill + the decoded token), {cores} threads")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name + " + state init + 1 decode token", "sample_tokens_per_head": Ts + 1},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU arm

def run_ours(args, rank, world, local_rank):
    import torch

    import recurrent_state_02_gb300 as la
    from recurrent_state_02_gb300 import _native, build as native_build
    from recurrent_state_02_gb300 import workloads as W

    native_build.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
    stream = torch.cuda.Stream(dev)
    L = _native.lib()

    w = W.UNGATED
    B, H, T, r, dv = w.B, w.H, w.T, w.r, w.dv
    base = W.prefill_inputs(w, seed=w.seed + 1000 * rank)
    dec = W.decode_inputs(W.DECODE.with_(B=B, H=H), seed=w.seed + 7 + 1000 * rank)
    sets = []
    for i in range(N_ROT):
        s = dict(q=base["q"].to(dev), k=base["k"].to(dev), v=base["v"].to(dev),
                 y=torch.empty((B, H, T, dv), device=dev, dtype=torch.bfloat16),
                 S=torch.empty((B, H, r, dv), device=dev, dtype=torch.float32),
                 z=torch.empty((B, H, r), device=dev, dtype=torch.float32),
                 qd=dec["q"].to(dev), kd=dec["k"].to(dev), vd=dec["v"].to(dev),
                 yd=torch.empty((B, H, 1, dv), device=dev, dtype=torch.bfloat16))
        sets.append(s)
    sh = stream.cuda_stream
    P = lambda t: t.data_ptr()
    # scratch of the segmented prefill (zero bytes when the plan does not split
    # sequences); the launches of one step run in order on one stream, so the
    # sets share it
    ws_bytes = int(L.la_prefill_workspace_bytes(B, H, T, r, dv, w.chunk))
    ws = torch.empty(max(ws_bytes, 256), device=dev, dtype=torch.uint8)

    def k_init(s):
        _native.check(L.la_state_init(P(s["S"]), P(s["z"]), B, H, r, dv, sh), "la_state_init")

    def k_prefill(s):
        _native.check(L.la_prefill_chunked(P(s["q"]), P(s["k"]), P(s["v"]), _native.LA_DTYPE_BF16, None,
                                           P(s["S"]), P(s["z"]), B, H, T, r, dv, w.chunk, w.eps, P(s["y"]),
                                           P(s["S"]), P(s["z"]), P(ws), ws_bytes, sh), "la_prefill_chunked")

    def k_decode(s):
        _native.check(L.la_decode_step(P(s["qd"]), P(s["kd"]), P(s["vd"]), _native.LA_DTYPE_BF16, None, P(s["S"]),
                                       P(s["z"]), B, H, r, dv, w.eps, P(s["yd"]), sh), "la_decode_step")

    # eager run once (sets kernel attributes, checks status), then capture graphs
    with torch.cuda.stream(stream):
        for s in sets:
            k_init(s); k_prefill(s); k_decode(s)
    assert _native.lib().la_last_device_status(sh) == 0
    step_graphs, prefill_graphs = [], []
    for s in sets:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            k_init(s); k_prefill(s); k_decode(s)
        step_graphs.append(g)
        g2 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g2, stream=stream):
            k_prefill(s)
        prefill_graphs.append(g2)
    # state init, (state pass, scan,) chunk kernel, decode
    prefill_launches = 3 if ws_bytes else 1
    launches_per_step = 2 + prefill_launches

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)

    def timed(graphs, K, W_):
        with torch.cuda.stream(stream):
            for i in range(W_):
                graphs[i % N_ROT].replay()
            barrier()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for i in range(K):
                graphs[i % N_ROT].replay()
            e1.record(stream)
            barrier()
        return e0.elapsed_time(e1) / 1e3  # seconds

    peak, peak_kind = read_peaks()
    with ClockSampler(gpu_index(local_rank)) as clk:
        # extra warm-up so the clock sampler sees the GPU under load
        t_start = time.time()
        with torch.cuda.stream(stream):
            n = 0
            while time.time() - t_start < args.clock_warmup_seconds or n < args.warmup:
                step_graphs[n % N_ROT].replay()
                n += 1
                if n % 50 == 0:
                    torch.cuda.synchronize(dev)
        torch.cuda.synchronize(dev)
        t0 = time.time()
        step_s = timed(step_graphs, args.steps, args.warmup)
        t1 = time.time()
        prefill_s = timed(prefill_graphs, args.steps, args.warmup)
    clocks = clk.summary(t0, t1)
    assert _native.lib().la_last_device_status(sh) == 0

    # max over ranks
    step_s, prefill_s = reduce_max([step_s, prefill_s], dev, dist)
    tokens_per_step = B * (T + 1)
    value = whole_job_rate(tokens_per_step, world, args.steps, step_s)
    ms_per_step = step_s / args.steps * 1e3
    pre_bytes = prefill_bytes(B, H, T, r, dv, with_state_in=True)
    pre_launch = prefill_s / args.steps
    achieved = pre_bytes / pre_launch / 1e9
    src = kernel_sources("prefill_tc.cu")
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "traffic": profile_traffic("prefill_tc_kernel<false, 64>", "B4 H16 T4096", src),
                "kernel": "prefill_tc_kernel<false, 64> (ungated, two 64-column CTAs per head)" + (
                    " timed with its state pass and scan (the sequences are split into a short first "
                    "segment and a long rest)" if ws_bytes else ""),
                "launches_per_prefill": prefill_launches, "algorithmic_bytes_per_launch": pre_bytes,
                "launch_us": pre_launch * 1e6, "peak_kind": peak_kind,
                "prefill_tokens_per_s": B * T * world / pre_launch,
                "prefill_token_heads_per_s": B * H * T * world / pre_launch,
                "tflops": prefill_flops(B, H, T, r, dv, w.chunk) / pre_launch / 1e12}

    only = set(args.only.split(",")) if args.only else None
    want = lambda name: only is None or name in only
    decode = delta = backward = e2e = None
    alu_peak = fp32_alu_peak_tflops(torch.cuda.get_device_properties(dev).multi_processor_count)

    if want("decode"):
        # decode on its own workload: B=256, H=16, state 256 MiB (> L2), in place
        dw = W.DECODE
        dinp = W.decode_inputs(dw, seed=dw.seed + 1000 * rank)
        dd = {k: (v.to(dev) if v is not None else None) for k, v in dinp.items()}
        ydec = torch.empty((dw.B, dw.H, 1, dw.dv), device=dev, dtype=torch.bfloat16)

        def k_dec_big():
            _native.check(L.la_decode_step(P(dd["q"]), P(dd["k"]), P(dd["v"]), _native.LA_DTYPE_BF16, None, P(dd["S"]),
                                           P(dd["z"]), dw.B, dw.H, dw.r, dw.dv, dw.eps, P(ydec), sh), "decode")

        with torch.cuda.stream(stream):
            k_dec_big()
        gd = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gd, stream=stream):
            k_dec_big()
        dec_s = timed([gd] * N_ROT, args.steps, args.warmup)
        dec_s, = reduce_max([dec_s], dev, dist)
        dbytes = decode_bytes(dw.B, dw.H, dw.r, dw.dv)
        dec_launch = dec_s / args.steps
        dec_gbs = dbytes / dec_launch / 1e9
        decode = {"workload": dw.name, "gb_per_s": dec_gbs * world, "per_gpu_gb_per_s": dec_gbs,
                  "frac_of_hbm_peak": dec_gbs / peak, "launch_us": dec_launch * 1e6,
                  "algorithmic_bytes_per_launch": dbytes, "tokens_per_s": dw.B * world / dec_launch,
                  "traffic": profile_traffic("decode128_kernel<true>", "B256 H16", kernel_sources("decode.cu"))}
        del dd, ydec, gd

        # a short continuation (8 tokens per request from the carried state, gated):
        # la_prefill_chunked in place, which takes the state-resident token walk
        cw = W.SHORT
        cin = {k: (v.to(dev) if v is not None else None)
               for k, v in W.prefill_inputs(cw, with_state=True, seed=cw.seed + 1000 * rank).items()}
        ycont = torch.empty((cw.B, cw.H, cw.T, cw.dv), device=dev, dtype=torch.bfloat16)

        def k_cont():
            _native.check(L.la_prefill_chunked(P(cin["q"]), P(cin["k"]), P(cin["v"]), _native.LA_DTYPE_BF16,
                                               P(cin["alpha"]), P(cin["S0"]), P(cin["z0"]), cw.B, cw.H, cw.T, cw.r,
                                               cw.dv, cw.chunk, cw.eps, P(ycont), P(cin["S0"]), P(cin["z0"]), None, 0,
                                               sh), "la_prefill_chunked (short)")

        with torch.cuda.stream(stream):
            k_cont()
        gc = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gc, stream=stream):
            k_cont()
        c_s = timed([gc] * N_ROT, args.steps, args.warmup)
        c_s, = reduce_max([c_s], dev, dist)
        assert _native.lib().la_last_device_status(sh) == 0
        c_launch = c_s / args.steps
        cbytes = short_bytes(cw.B, cw.H, cw.T, cw.r, cw.dv, cw.gated)
        c_gbs = cbytes / c_launch / 1e9
        decode["short_continuation"] = {
            "workload": cw.name, "entry": "la_prefill_chunked (T <= 32: the state-resident token walk)",
            "launch_us": c_launch * 1e6, "tokens_per_s": cw.B * cw.T * world / c_launch,
            "token_heads_per_s": cw.B * cw.H * cw.T * world / c_launch,
            "roofline": {"bound": "hbm", "achieved": c_gbs, "peak": peak, "unit": "GB/s", "frac": c_gbs / peak,
                         "peak_kind": peak_kind, "algorithmic_bytes_per_launch": cbytes,
                         "traffic": profile_traffic("decode128_multi_kernel<true>", "B256 H16 T8",
                                                    kernel_sources("decode.cu"))}}
        del cin, ycont, gc

    # the gated (B2 H16 T16384, alpha = sigmoid(N(3,1))) and long (B1 H32 T65536,
    # sigma = 2) prefill workloads, each on its own inputs from a zero state: the
    # whole la_prefill_chunked call (state pass, scan and chunk kernel when the
    # sequences are split into segments) replayed as a CUDA graph; two input sets
    # of 270 MB alternate for the gated workload, the long one's 2.1 GB set
    # exceeds L2 by itself
    def prefill_workload(pw, nsets, kernel):
        pin = W.prefill_inputs(pw, seed=pw.seed + 1000 * rank)
        psets = []
        for _ in range(nsets):
            psets.append(dict(q=pin["q"].to(dev), k=pin["k"].to(dev), v=pin["v"].to(dev),
                              alpha=pin["alpha"].to(dev) if pin["alpha"] is not None else None,
                              y=torch.empty((pw.B, pw.H, pw.T, pw.dv), device=dev, dtype=torch.bfloat16),
                              S=torch.empty((pw.B, pw.H, pw.r, pw.dv), device=dev, dtype=torch.float32),
                              z=torch.empty((pw.B, pw.H, pw.r), device=dev, dtype=torch.float32)))
        del pin
        nws = int(L.la_prefill_workspace_bytes(pw.B, pw.H, pw.T, pw.r, pw.dv, pw.chunk))
        pws = torch.empty(max(nws, 256), device=dev, dtype=torch.uint8)

        def call(s):
            _native.check(L.la_prefill_chunked(P(s["q"]), P(s["k"]), P(s["v"]), _native.LA_DTYPE_BF16,
                                               P(s["alpha"]) if s["alpha"] is not None else None, None, None,
                                               pw.B, pw.H, pw.T, pw.r, pw.dv, pw.chunk, pw.eps, P(s["y"]),
                                               P(s["S"]), P(s["z"]), P(pws), nws, sh), "la_prefill_chunked")

        graphs = []
        for s in psets:
            with torch.cuda.stream(stream):
                call(s)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                call(s)
            graphs.append(g)
        t_s = timed([graphs[i % nsets] for i in range(N_ROT)], args.steps, args.warmup)
        t_s, = reduce_max([t_s], dev, dist)
        assert _native.lib().la_last_device_status(sh) == 0
        t_call = t_s / args.steps
        nbytes = prefill_bytes(pw.B, pw.H, pw.T, pw.r, pw.dv, with_state_in=False) + (
            pw.B * pw.H * pw.T * 4 if pw.gated else 0)
        gbs = nbytes / t_call / 1e9
        del psets, graphs, pws
        torch.cuda.empty_cache()
        return {"workload": pw.name, "call_us": t_call * 1e6, "tokens_per_s": pw.B * pw.T * world / t_call,
                "token_heads_per_s": pw.B * pw.H * pw.T * world / t_call,
                "tflops": prefill_flops(pw.B, pw.H, pw.T, pw.r, pw.dv, pw.chunk) / t_call / 1e12,
                "launches_per_call": 3 if nws else 1,
                "l2": f"{nsets} input set(s) of {nbytes / 1e6:.0f} MB (> 129 MB L2)",
                "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                             "peak_kind": peak_kind,
                             "timed": "the whole call" + (" (state pass, scan and chunk kernel)" if nws else ""),
                             "kernel": kernel, "algorithmic_bytes_per_launch": nbytes,
                             "traffic": profile_traffic(kernel, f"B{pw.B} H{pw.H} T{pw.T}",
                                                        kernel_sources("prefill_tc.cu"))}}

    gated_prefill = prefill_workload(W.GATED, 2, "prefill_tc_kernel<true, 128>") if want("gated") else None
    long_prefill = prefill_workload(W.LONG, 1, "prefill_tc_kernel<false, 128>") if want("long") else None

    varlen = None
    if want("varlen"):
        # packed serving batches through la_prefill_varlen: two prompt mixes from zero
        # states (q, k, v of 497 MB and 1.1 GB, > L2), and ragged short continuations
        # from 256 x 16 carried states in place (270 MB of state, > L2): the whole
        # call (the token walk, the plan, state pass, scan and chunk kernel)
        # replayed as a CUDA graph
        varlen = {}
        for vw in (W.VARLEN_LONG, W.VARLEN_LOGU, W.VARLEN_SHORT):
            vin = W.varlen_inputs(vw, device=dev, seed=vw.seed + 1000 * rank)
            nvb = len(vw.lens)
            yv = torch.empty((vw.T, vw.H, vw.dv), device=dev, dtype=torch.bfloat16)
            Sv = torch.empty((nvb, vw.H, vw.r, vw.dv), device=dev, dtype=torch.float32)
            zv = torch.empty((nvb, vw.H, vw.r), device=dev, dtype=torch.float32)
            nvws = int(L.la_prefill_varlen_workspace_bytes(nvb, vw.H, vw.T, vw.r, vw.dv))
            vws = torch.empty(max(nvws, 256), device=dev, dtype=torch.uint8)

            # carried states are updated in place (S0 = S_out), as a serving step would
            if "S0" in vin:
                Sv, zv = vin["S0"], vin["z0"]
            opt = lambda n: P(vin[n]) if n in vin else None

            def k_varlen():
                _native.check(L.la_prefill_varlen(P(vin["q"]), P(vin["k"]), P(vin["v"]), _native.LA_DTYPE_BF16,
                                                  opt("alpha"), opt("S0"), opt("z0"), P(vin["cu_seqlens"]), nvb, vw.H,
                                                  vw.T, vw.r, vw.dv, vw.chunk, vw.eps, P(yv), P(Sv), P(zv),
                                                  P(vws) if nvws else None, nvws, sh), "la_prefill_varlen")

            with torch.cuda.stream(stream):
                k_varlen()
            gv = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gv, stream=stream):
                k_varlen()
            v_s = timed([gv] * N_ROT, args.steps, args.warmup)
            v_s, = reduce_max([v_s], dev, dist)
            assert _native.lib().la_last_device_status(sh) == 0
            v_call = v_s / args.steps
            # the dominant kernel: the token walk for the short continuations, else the chunk kernel
            vkern, vsrc = (("decode128_multi_kernel<true, 2, packed>", "decode.cu") if vw is W.VARLEN_SHORT
                           else ("prefill_tc_kernel<false, 128> items", "prefill_tc.cu"))
            vbytes = varlen_bytes(nvb, vw.H, vw.T, vw.r, vw.dv) + (
                nvb * vw.H * 4 * (vw.r * vw.dv + vw.r) if "S0" in vin else 0) + (vw.T * vw.H * 4 if vw.gated else 0)
            v_gbs = vbytes / v_call / 1e9
            varlen[vw.name] = {
                "call_us": v_call * 1e6, "tokens_per_s": vw.T * world / v_call,
                "token_heads_per_s": vw.T * vw.H * world / v_call, "sequences": nvb, "tokens": vw.T,
                "longest": max(vw.lens), "launches_per_call": 5 if nvws else 1,   # walk, plan, state pass, scan, chunk kernel
                "roofline": {"bound": "hbm", "achieved": v_gbs, "peak": peak, "unit": "GB/s", "frac": v_gbs / peak,
                             "peak_kind": peak_kind, "algorithmic_bytes_per_launch": vbytes,
                             "timed": "the whole call", "kernel": vkern,
                             "traffic": profile_traffic(vkern, f"B{nvb} H{vw.H} T{vw.T}", kernel_sources(vsrc))}}
            del vin, yv, Sv, zv, vws, gv
        torch.cuda.empty_cache()

    if want("delta"):
        # delta-rule memory on its own workload (B=4, H=16, T=4096, r = dv = 128, BF16;
        # q, k, v 201 MB > L2): the chunked tensor-core entry point (its two launches,
        # T of every chunk and then the state chain) and the FP32 token recurrence,
        # each replayed as a CUDA graph
        xw = W.DELTA
        xin = {k: (v.to(dev) if v is not None else None) for k, v in W.delta_inputs(xw, seed=xw.seed + 1000 * rank).items()}
        ydel = torch.empty((xw.B, xw.H, xw.T, xw.dv), device=dev, dtype=torch.bfloat16)
        Sdel = torch.empty((xw.B, xw.H, xw.r, xw.dv), device=dev, dtype=torch.float32)
        xws_bytes = _native.lib().la_delta_chunked_workspace_bytes(xw.B, xw.H, xw.T)
        xws = torch.empty(xws_bytes, device=dev, dtype=torch.uint8)

        def k_delta_tc():
            _native.check(L.la_delta_rule_chunked(P(xin["q"]), P(xin["k"]), P(xin["v"]), _native.LA_DTYPE_BF16,
                                                  P(xin["beta"]), None, xw.B, xw.H, xw.T, xw.r, xw.dv, P(ydel), P(Sdel),
                                                  P(xws), xws_bytes, sh), "la_delta_rule_chunked")

        def k_delta():
            _native.check(L.la_delta_rule(P(xin["q"]), P(xin["k"]), P(xin["v"]), _native.LA_DTYPE_BF16, P(xin["beta"]),
                                          None, xw.B, xw.H, xw.T, xw.r, xw.dv, P(ydel), P(Sdel), sh), "la_delta_rule")

        x_times = []
        for fn in (k_delta_tc, k_delta):
            with torch.cuda.stream(stream):
                fn()
            gx = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gx, stream=stream):
                fn()
            x_times.append(timed([gx] * N_ROT, args.steps, args.warmup))
        xc_s, x_s = reduce_max(x_times, dev, dist)
        assert _native.lib().la_last_device_status(sh) == 0
        xc_launch, x_launch = xc_s / args.steps, x_s / args.steps
        xbytes = delta_bytes(xw.B, xw.H, xw.T, xw.r, xw.dv)
        xc_gbs = xbytes / xc_launch / 1e9
        x_tflops = delta_flops(xw.B, xw.H, xw.T, xw.r, xw.dv) / x_launch / 1e12
        delta = {"workload": xw.name, "entry": "la_delta_rule_chunked", "launch_us": xc_launch * 1e6,
                 "tokens_per_s": xw.B * xw.T * world / xc_launch,
                 "roofline": {"bound": "hbm", "achieved": xc_gbs, "peak": peak, "unit": "GB/s",
                              "frac": xc_gbs / peak, "peak_kind": peak_kind,
                              "timed": "the whole call (both launches)",
                              "traffic": profile_traffic("delta_tc_kernel", "B4 H16 T4096",
                                                         kernel_sources("delta_tc.cu")),
                              "algorithmic_bytes_per_launch": xbytes},
                 "token_recurrence": {
                     "entry": "la_delta_rule", "launch_us": x_launch * 1e6,
                     "tokens_per_s": xw.B * xw.T * world / x_launch,
                     "roofline": {"bound": "alu", "achieved": x_tflops, "peak": alu_peak, "unit": "TFLOP/s",
                                  "frac": x_tflops / alu_peak, "peak_kind": "nominal FP32 FMA (SMs x 128 x 2 x max clock)",
                                  "traffic": profile_traffic("delta_kernel<bf16,128>", "B4 H16 T4096",
                                                             kernel_sources("delta.cu")),
                                  "algorithmic_flops_per_launch": delta_flops(xw.B, xw.H, xw.T, xw.r, xw.dv)}}}

    if want("backward"):
        # backward pass on the gated shape of the prefill (B=4, H=16, T=4096, BF16,
        # alpha = sigmoid(N(3,1))): its five launches replayed as one CUDA graph
        bw = W.UNGATED.with_(gated=True)
        bin_ = {k: (v.to(dev) if v is not None else None)
                for k, v in W.prefill_inputs(bw, seed=bw.seed + 11 + 1000 * rank).items()}
        ybw = torch.empty((bw.B, bw.H, bw.T, bw.dv), device=dev, dtype=torch.bfloat16)
        Sbw = torch.empty((bw.B, bw.H, bw.r, bw.dv), device=dev, dtype=torch.float32)
        zbw = torch.empty((bw.B, bw.H, bw.r), device=dev, dtype=torch.float32)
        dybw = torch.randn((bw.B, bw.H, bw.T, bw.dv), generator=torch.Generator().manual_seed(bw.seed + 12)).to(dev,
                                                                                                                  torch.bfloat16)
        gq, gk, gv = (torch.empty_like(bin_[n]) for n in ("q", "k", "v"))
        ga = torch.empty((bw.B, bw.H, bw.T), device=dev, dtype=torch.float32)
        gS0 = torch.empty((bw.B, bw.H, bw.r, bw.dv), device=dev, dtype=torch.float32)
        gz0 = torch.empty((bw.B, bw.H, bw.r), device=dev, dtype=torch.float32)
        wsb = torch.empty(int(L.la_backward_workspace_bytes(bw.B, bw.H, bw.T)), device=dev, dtype=torch.uint8)

        def k_backward():
            _native.check(L.la_prefill_backward(P(bin_["q"]), P(bin_["k"]), P(bin_["v"]), _native.LA_DTYPE_BF16,
                                                P(bin_["alpha"]), None, None, bw.B, bw.H, bw.T, bw.r, bw.dv, bw.eps,
                                                P(ybw), P(dybw), None, None, P(gq), P(gk), P(gv), P(ga), P(gS0), P(gz0),
                                                P(wsb), wsb.numel(), sh), "la_prefill_backward")

        # the same backward with what a training forward keeps: the denominators (no
        # z pass) and the states entering the backward's segments (no forward state pass)
        dbw = torch.empty((bw.B, bw.H, bw.T), device=dev, dtype=torch.float32)
        nstb = int(L.la_backward_states_bytes(bw.B, bw.H, bw.T))
        stbw = torch.empty(max(1, nstb // 4), device=dev, dtype=torch.float32)
        pst = P(stbw) if nstb else None

        def k_backward_saved():
            _native.check(L.la_prefill_backward_saved(P(bin_["q"]), P(bin_["k"]), P(bin_["v"]), _native.LA_DTYPE_BF16,
                                                      P(bin_["alpha"]), None, None, bw.B, bw.H, bw.T, bw.r, bw.dv,
                                                      P(ybw), P(dybw), P(dbw), pst, None, None, P(gq), P(gk), P(gv),
                                                      P(ga), P(gS0), P(gz0), P(wsb), wsb.numel(), sh),
                          "la_prefill_backward_saved")

        with torch.cuda.stream(stream):
            _native.check(L.la_prefill_chunked_save(P(bin_["q"]), P(bin_["k"]), P(bin_["v"]), _native.LA_DTYPE_BF16,
                                                    P(bin_["alpha"]), None, None, bw.B, bw.H, bw.T, bw.r, bw.dv,
                                                    bw.chunk, bw.eps, P(ybw), P(Sbw), P(zbw), P(dbw), pst, None, 0,
                                                    sh),
                          "la_prefill_chunked_save")
            k_backward()
            k_backward_saved()
        gb = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gb, stream=stream):
            k_backward()
        gbs = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gbs, stream=stream):
            k_backward_saved()
        bsteps = max(1, min(args.steps, 20))
        b_s = timed([gb] * N_ROT, bsteps, max(3, min(args.warmup, 3)))
        bs_s = timed([gbs] * N_ROT, bsteps, max(3, min(args.warmup, 3)))
        b_s, bs_s = reduce_max([b_s, bs_s], dev, dist)
        assert _native.lib().la_last_device_status(sh) == 0
        b_call, bs_call = b_s / bsteps, bs_s / bsteps
        b_bytes = backward_bytes(bw.B, bw.H, bw.T, bw.r, bw.dv, True)
        bs_bytes = b_bytes + 4 * bw.B * bw.H * bw.T + nstb   # and the saved d_t and states read
        b_gbs = b_bytes / b_call / 1e9
        backward = {"workload": bw.name.replace("prefill", "backward of the gated prefill,"), "call_us": b_call * 1e6,
                    "launches_per_call": 12, "tokens_per_s": bw.B * bw.T * world / b_call, "steps": bsteps,
                    "roofline": {"bound": "hbm", "achieved": b_gbs, "peak": peak, "unit": "GB/s",
                                 "frac": b_gbs / peak, "peak_kind": peak_kind, "scope": "whole call",
                                 "algorithmic_bytes_per_call": b_bytes,
                                 "tensor_tflops": backward_flops(bw.B, bw.H, bw.T, bw.r, bw.dv, True) / b_call / 1e12,
                                 "algorithmic_flops_per_call": backward_flops(bw.B, bw.H, bw.T, bw.r, bw.dv, True)},
                    "saved_d": {"entry": "la_prefill_backward_saved (d_t and the segment states from "
                                         "la_prefill_chunked_save)",
                                "call_us": bs_call * 1e6, "launches_per_call": 9 - (2 if nstb else 0),
                                "tokens_per_s": bw.B * bw.T * world / bs_call,
                                "roofline": {"bound": "hbm", "achieved": bs_bytes / bs_call / 1e9, "peak": peak,
                                             "unit": "GB/s", "frac": bs_bytes / bs_call / 1e9 / peak,
                                             "peak_kind": peak_kind, "scope": "whole call",
                                             "algorithmic_bytes_per_call": bs_bytes}}}

    if want("e2e"):
        # end to end through the public API with host buffers (pinned), every step:
        # H2D of q, k, v (+ the decode token), the three calls, D2H of y, S, z, y_decode.
        # Steps are pipelined as a serving loop would run them: the copies in of step
        # i+1 and the copies out of step i-1 run on their own streams while step i
        # computes.  Two device buffer sets (and two pinned host output sets)
        # alternate; events order every reuse of a buffer after its last reader.
        hq, hk, hv = (base[n].pin_memory() for n in ("q", "k", "v"))
        hqd, hkd, hvd = (dec[n].pin_memory() for n in ("q", "k", "v"))
        hout = [dict(y=torch.empty((B, H, T, dv), dtype=torch.bfloat16).pin_memory(),
                     S=torch.empty((B, H, r, dv), dtype=torch.float32).pin_memory(),
                     z=torch.empty((B, H, r), dtype=torch.float32).pin_memory(),
                     yd=torch.empty((B, H, 1, dv), dtype=torch.bfloat16).pin_memory()) for _ in range(2)]
        h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hqd, hkd, hvd))
        d2h = sum(t.numel() * t.element_size() for t in hout[0].values())
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev = {n: [torch.cuda.Event(), torch.cuda.Event()] for n in ("in", "comp", "out")}

        def e2e_step(i):
            b = i % 2
            s, ho = sets[b], hout[b]
            with torch.cuda.stream(s_in):          # inputs of step i, once step i-2 stopped reading them
                if i >= 2:
                    s_in.wait_event(ev["comp"][b])
                s["q"].copy_(hq, non_blocking=True); s["k"].copy_(hk, non_blocking=True)
                s["v"].copy_(hv, non_blocking=True); s["qd"].copy_(hqd, non_blocking=True)
                s["kd"].copy_(hkd, non_blocking=True); s["vd"].copy_(hvd, non_blocking=True)
                ev["in"][b].record(s_in)
            with torch.cuda.stream(stream):        # the step, once its inputs are in and step i-2 was read back
                stream.wait_event(ev["in"][b])
                if i >= 2:
                    stream.wait_event(ev["out"][b])
                S, z = la.state_init(B, H, r, dv, S=s["S"], z=s["z"])
                la.prefill_chunked(s["q"], s["k"], s["v"], S0=S, z0=z, S_out=S, z_out=z, y=s["y"], chunk=w.chunk,
                                   eps=w.eps)
                la.decode_step(s["qd"], s["kd"], s["vd"], S, z, eps=w.eps, y=s["yd"])
                ev["comp"][b].record(stream)
            with torch.cuda.stream(s_out):         # its results back to the host
                s_out.wait_event(ev["comp"][b])
                ho["y"].copy_(s["y"], non_blocking=True); ho["S"].copy_(s["S"], non_blocking=True)
                ho["z"].copy_(s["z"], non_blocking=True); ho["yd"].copy_(s["yd"], non_blocking=True)
                ev["out"][b].record(s_out)

        e2e_steps = max(1, min(args.steps, 50))
        n_warm = max(2, min(args.warmup, 5))
        for i in range(n_warm):
            e2e_step(i)
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s_in)
        for i in range(n_warm, n_warm + e2e_steps):
            e2e_step(i)
        e1.record(s_out)
        barrier()
        e2e_s = e0.elapsed_time(e1) / 1e3
        e2e_s, = reduce_max([e2e_s], dev, dist)
        assert _native.lib().la_last_device_status(sh) == 0
        e2e = {"value": whole_job_rate(tokens_per_step, world, e2e_steps, e2e_s), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": e2e_steps, "ms_per_step": e2e_s / e2e_steps * 1e3,
               "pipelining": "copies in (step i+1), compute (step i) and copies out (step i-1) on three streams"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tps, cores, desc, _ = oracle_tokens_per_s(w, args.cpu_seconds)
        cpu = {"value": tps, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": desc}
        # the oracles of the delta rule and of the backward, beside their GPU figures
        if delta is not None:
            delta["cpu_baseline"] = oracle_rate("delta", xw, args.cpu_seconds / 4)
        for entry, pw in ((gated_prefill, W.GATED), (long_prefill, W.LONG)):
            if entry is None:
                continue
            tps_p, cores_p, desc_p, _ = oracle_tokens_per_s(pw, args.cpu_seconds / 4)
            entry["cpu_baseline"] = {"value": tps_p, "unit": "tokens/s", "cores": cores_p, "kind": "oracle",
                                     "sample": desc_p}
        if backward is not None:
            backward["cpu_baseline"] = oracle_rate("backward", bw, args.cpu_seconds / 4)

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": {"workload": w.name + " + state init + 1 decode token per request",
                           "B": B, "H": H, "T": T, "r": r, "dv": dv, "chunk": w.chunk, "tokens_per_step": tokens_per_step,
                           "l2": f"{N_ROT} rotating input/output sets of "
                                 f"{prefill_bytes(B, H, T, r, dv) / 1e6:.0f} MB (> 129 MB L2)",
                           "parallelism": f"replicas x{world} (independent batches, no collective)",
                           "launch": "CUDA graph per step"},
                "roofline": roofline, "decode": decode, "gated_prefill": gated_prefill, "long_prefill": long_prefill,
                "varlen": varlen,
                "delta_rule": delta, "backward": backward, "cpu_baseline": cpu,
                "e2e": e2e,
                "gpu_launches": launches_per_step * args.steps, "clocks": clocks}
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    # 2000 steps of the headline (about 0.4 s timed with its prefill) give the clock
    # sampler several readings inside the timed region
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", default="",
                    help="comma-separated subset of the extra workloads to run beside the step: "
                         "decode,gated,long,varlen,delta,backward,e2e (default: all)")
    ap.add_argument("--clock-warmup-seconds", type=float, default=0.6,
                    help="untimed load before timing so that clock samples see the GPU busy (0 under a profiler)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus:
        ap.error(f"--gpus {args.gpus} but WORLD_SIZE={world}")
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
