"""Benchmark of the exact attention forward on one or more B300s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step is one attn_fwd call (the whole forward: scores, mask, online softmax, P.V,
epilogue) over one batch of the named workload, inputs already resident in HBM.
Under torchrun every rank runs its own full batch (seed + rank) on its own GPU: the
work is independent per (batch, head), so the ranks never exchange data, and the
scaling is weak. Rank 0 prints one JSON line.

Timing: W untimed warm-up calls, then K timed calls, bracketed by a barrier and a
device synchronisation on both sides. A 256 MiB buffer (more than the 126 MB L2) is
written and then read back before every call, leaving L2 with clean lines of it,
and each call is timed by its own pair of CUDA events on the launching stream, so
the flush is not counted. value = algorithmic
FLOPs of all ranks / the slowest rank's summed kernel time; FLOPs are 4 * d per
visible (query, key) pair, masked pairs not counted.

--impl reference times the fp64 CPU oracle on this host's cores over bounded
samples of the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from exact_self_attention_fwd_b300.inputs import (DECODE_WORKLOADS, WORKLOADS, DecodeWorkload,  # noqa: E402
                                                   Workload, make_qkv, make_qkv_decode)

DEFAULT_WORKLOAD = "gqa_8k"
FLUSH_BYTES = 256 << 20


def flush_l2(buf):
    """Evict L2 before a timed call: write the 256 MiB buffer (about twice the L2), then
    read it back, so that L2 ends up holding clean lines of it; the timed call then
    neither hits its own inputs in L2 nor pays for writing back the flush's dirty
    lines."""
    buf.zero_()
    buf.view(-1, 4096).max(dim=1)
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
KERNEL_SOURCES = ["exact_self_attention_fwd_b300/csrc/attn_fwd.cu",
                  "exact_self_attention_fwd_b300/csrc/ptx.cuh"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.txt")


# ------------------------------------------------------------------ accounting
def visible_pairs(N: int, causal: bool, window: int) -> int:
    """Number of (i, j) with key j visible to query i, per (batch, query head)."""
    if not causal:
        return N * N
    if window <= 0 or window >= N:
        return N * (N + 1) // 2
    # rows i < W see i + 1 keys, rows i >= W see W keys
    return window * (window + 1) // 2 + (N - window) * window


def flops(w: Workload) -> int:
    return 4 * w.B * w.Hq * visible_pairs(w.N, w.causal, w.window) * w.d


def bwd_flops(w: Workload) -> int:
    """FLOPs of one backward pass over the visible pairs: five products of d MACs per
    pair (S and dP recomputed, then dV, dK and dQ), 2.5 times the forward's."""
    return 10 * w.B * w.Hq * visible_pairs(w.N, w.causal, w.window) * w.d


def hbm_bytes(w: Workload) -> int:
    """Algorithmic bytes: Q, K, V read once (bf16), O written (bf16), LSE written (fp32)."""
    q = w.B * w.Hq * w.N * w.d * 2
    kv = 2 * w.B * w.Hkv * w.N * w.d * 2
    return q + kv + q + w.B * w.Hq * w.N * 4


def decode_flops(w: DecodeWorkload) -> int:
    """4 d per visible (query, key) pair; query i stands at position i + Nk - Nq."""
    pairs = 0
    for i in range(w.Nq):
        pos = i + w.Nk - w.Nq
        pairs += (pos + 1) if w.causal else w.Nk
    return 4 * w.B * w.Hq * pairs * w.d


def decode_hbm_bytes(w: DecodeWorkload) -> int:
    """Q, K, V read once (bf16), O written (bf16), LSE written (fp32)."""
    q = w.B * w.Hq * w.Nq * w.d * 2
    return 2 * q + 2 * w.B * w.Hkv * w.Nk * w.d * 2 + w.B * w.Hq * w.Nq * 4


def kernel_sha() -> str:
    """Hash of the source the forward kernel is built from: the device code of attn_fwd.cu
    up to the end of attn_fwd_kernel, the host function that launches it, and ptx.cuh.
    Edits elsewhere in the translation unit (other kernels, other entry points) leave
    it, and so a recorded traffic figure, unchanged."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            src = f.read()
        if rel.endswith("attn_fwd.cu"):
            end = src.find(b"// Block quantisation to e4m3")
            start = src.find(b"int launch(const void *q")
            stop = src.find(b"\n}\n", start) if start >= 0 else -1
            if end > 0 and start >= 0 and stop > start:
                src = src[:end] + src[start:stop]
        h.update(src)
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch from an ncu capture, if it was taken on the current kernel.

    profiles/traffic.txt lines: <workload> <bytes per launch> <kernel sha> <note...>
    """
    if not os.path.exists(TRAFFIC_FILE):
        return None
    sha = kernel_sha()
    with open(TRAFFIC_FILE) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 3 and not line.startswith("#") and parts[0] == workload and parts[2] == sha:
                return int(float(parts[1]))
    return None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ distributed
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int):
    """Control-plane group only (barrier, max over ranks): gloo on the host."""
    if world <= 1:
        return None
    import torch.distributed as dist
    if not dist.is_initialized():
        dist.init_process_group("gloo")
    return dist


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(dist, x: float) -> float:
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ clocks
CLOCK_QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
               "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def nvsmi_index(local_rank: int) -> str:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    ids = [x.strip() for x in vis.split(",") if x.strip()]
    if ids and local_rank < len(ids):
        return ids[local_rank]
    return str(local_rank)


class ClockSampler:
    """nvidia-smi sampling every 100 ms in a child process (our own PID, stopped by PID)."""

    def __init__(self, gpu: str, path: str):
        self.path = path
        self.proc = None
        try:
            self.f = open(path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", gpu, f"--query-gpu={CLOCK_QUERY}", "--format=csv,nounits",
                 "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self, t0: float, t1: float):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        with open(self.path) as f:
            rows = list(csv.reader(io.StringIO(f.read())))
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        head = [h.strip() for h in rows[0]]
        samples = []
        for r in rows[1:]:
            if len(r) != len(head):
                continue
            d = dict(zip(head, (x.strip() for x in r)))
            try:
                ts = time.mktime(time.strptime(d["timestamp"].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + d["timestamp"].split(".")[1]) if "." in d["timestamp"] else 0.0
            except (ValueError, KeyError, IndexError):
                continue
            samples.append((ts, d))
        inside = [d for ts, d in samples if t0 - 0.05 <= ts <= t1 + 0.05]
        use = inside if inside else [d for _, d in samples]

        def col(d, key):
            for k, v in d.items():
                if k.startswith(key):
                    return v
            return ""

        mhz = [float(col(d, "clocks.current.sm") or col(d, "clocks.sm") or "nan") for d in use]
        mhz = [m for m in mhz if m == m]
        mx = [float(col(d, "clocks.max.sm") or "nan") for d in use]
        reasons = set()
        for d in use:
            for key, name in (("clocks_event_reasons.hw_slowdown", "hw_slowdown"),
                              ("clocks_event_reasons.hw_thermal_slowdown", "hw_thermal_slowdown"),
                              ("clocks_event_reasons.sw_thermal_slowdown", "sw_thermal_slowdown"),
                              ("clocks_event_reasons.sw_power_cap", "sw_power_cap")):
                if col(d, key).lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(mhz) if mhz else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons),
                "samples_in_region": len(inside)}


# ------------------------------------------------------------------ oracle (CPU) timing
def oracle_sample(w: Workload, seconds: float, seed: int):
    """Time the fp64 oracle on a random sample of rows of workload w for about `seconds`.

    Returns (TFLOP/s, cores, description). Rows are drawn uniformly over every
    (batch, head, query); the FLOPs of a row are 4 * d * (its visible keys)."""
    import numpy as np
    import oracle

    q, k, v = make_qkv(w.B, w.Hq, w.Hkv, w.N, w.d, w.seed, w.q_head0_scale)
    cores = oracle.default_threads()
    rng = np.random.default_rng(seed)
    total_rows = w.B * w.Hq * w.N

    def row_flops(rows):
        i = rows % w.N
        if not w.causal:
            nvis = np.full(rows.shape, w.N, dtype=np.int64)
        else:
            nvis = i + 1
            if w.window > 0:
                nvis = np.minimum(nvis, w.window)
        return int(4 * w.d * nvis.sum())

    oracle.load()
    n = max(cores, 8)
    while True:
        rows = np.sort(rng.integers(0, total_rows, size=n)).astype(np.int64)
        t0 = time.perf_counter()
        oracle.attn_ref_rows(q, k, v, w.causal, w.window, w.scale, rows, nthreads=cores)
        dt = time.perf_counter() - t0
        if dt >= seconds or n >= total_rows:
            break
        n = min(total_rows, max(n * 2, int(n * seconds / max(dt, 1e-3) * 1.05)))
    return row_flops(rows) / dt / 1e12, cores, f"{n} random query rows of {total_rows} ({dt:.1f} s)"


# ------------------------------------------------------------------ arms
def run_reference(args, w: Workload):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    import numpy as np
    import oracle

    q, k, v = make_qkv(w.B, w.Hq, w.Hkv, w.N, w.d, w.seed, w.q_head0_scale)
    cores = oracle.default_threads()
    oracle.load()
    rng = np.random.default_rng(12345)
    total_rows = w.B * w.Hq * w.N
    budget = args.ref_seconds / max(1, args.steps + args.warmup)
    # calibrate rows per step so that all steps fit in the budget
    n = cores
    t0 = time.perf_counter()
    oracle.attn_ref_rows(q, k, v, w.causal, w.window, w.scale,
                         np.sort(rng.integers(0, total_rows, size=n)), nthreads=cores)
    per_row = (time.perf_counter() - t0) / n
    n = int(max(1, min(total_rows, budget / max(per_row, 1e-9))))

    def step():
        rows = np.sort(rng.integers(0, total_rows, size=n)).astype(np.int64)
        i = rows % w.N
        nvis = np.full(rows.shape, w.N) if not w.causal else (
            np.minimum(i + 1, w.window) if w.window > 0 else i + 1)
        t = time.perf_counter()
        oracle.attn_ref_rows(q, k, v, w.causal, w.window, w.scale, rows, nthreads=cores)
        return time.perf_counter() - t, int(4 * w.d * nvis.sum())

    for _ in range(args.warmup):
        step()
    tot_t, tot_f = 0.0, 0
    for _ in range(args.steps):
        dt, f = step()
        tot_t += dt
        tot_f += f
    value = tot_f / tot_t / 1e12
    line = {
        "impl": "reference", "metric": "attention fwd TFLOP/s (unmasked FLOPs)", "value": value,
        "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * tot_t / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,1) rounded to bf16)",
        "config": {"workload": w.name, "shape": w.note, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv,
                   "N": w.N, "d": w.d, "causal": w.causal, "window": w.window},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"{n} random query rows per step of {total_rows}"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def roofline_of(w: Workload, seconds_per_call: float, peaks: dict) -> dict:
    """The bound that limits workload w on this chip and the fraction of it achieved.

    Long sequences are tensor-core bound (FLOP/byte far above the ridge); the
    short-sequence bidirectional workload is HBM bound; the one-tile workload is bound
    by launch latency (its microseconds per call are the figure, no fraction)."""
    if w.name == "tiny":
        return {"bound": "latency", "achieved": seconds_per_call * 1e6, "peak": None, "unit": "us per call",
                "frac": None}
    if w.name == "vit_base":
        achieved = hbm_bytes(w) / seconds_per_call / 1e9
        peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
        return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak}
    achieved = flops(w) / seconds_per_call / 1e12
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    sustained = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    return {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
            "frac_vs_sustained": achieved / sustained}


def measure_workload(ea, w: Workload, dev, steps: int, warmup: int, seed_offset: int = 0, flush: bool = True):
    """Device time per attn_fwd call on workload w (seconds).

    Calls of at least a few microseconds are timed one by one with CUDA events, a
    256 MiB write-then-read between them flushing L2. The tiny workload's call is shorter
    than the host's launch overhead, so there a CUDA graph of `steps` calls is
    replayed and timed as a whole (its 66 KB of inputs stay in L2)."""
    import torch
    q, k, v = make_qkv(w.B, w.Hq, w.Hkv, w.N, w.d, w.seed + seed_offset, w.q_head0_scale)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    out = torch.empty_like(qd)
    lse = torch.empty((w.B, w.Hq, w.N), dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(dev)

    def call():
        ea.attn_fwd(qd, kd, vd, causal=w.causal, window=w.window, scale=w.scale, out=out, lse=lse,
                    stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            call()
    torch.cuda.synchronize(dev)
    if flops(w) < 1e8:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for _ in range(steps):
                ea.attn_fwd(qd, kd, vd, causal=w.causal, window=w.window, scale=w.scale, out=out,
                            lse=lse, stream=torch.cuda.current_stream(dev))
        g.replay()
        torch.cuda.synchronize(dev)
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        with torch.cuda.stream(stream):
            g.replay()
        s1.record(stream)
        torch.cuda.synchronize(dev)
        per = s0.elapsed_time(s1) / 1e3 / steps
        return per, "CUDA graph of %d calls" % steps
    buf = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev) if flush else None
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    with torch.cuda.stream(stream):
        for i in range(steps):
            if flush:
                flush_l2(buf)
            starts[i].record(stream)
            call()
            ends[i].record(stream)
    torch.cuda.synchronize(dev)
    per = sum(a.elapsed_time(b) for a, b in zip(starts, ends)) / 1e3 / steps
    return per, ("per-call CUDA events, L2 flushed between calls" if flush
                 else "per-call CUDA events, calls back to back (no flush)")


def measure_decode(ea, w: DecodeWorkload, dev, steps: int, warmup: int, seed_offset: int = 0):
    """Device time per attn_fwd_decode call (seconds), per-call CUDA events, L2 flushed
    between calls; the split workspace is allocated once, outside the timed calls."""
    import torch
    q, k, v = make_qkv_decode(w.B, w.Hq, w.Hkv, w.Nq, w.Nk, w.d, w.seed + seed_offset)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    out = torch.empty_like(qd)
    lse = torch.empty((w.B, w.Hq, w.Nq), dtype=torch.float32, device=dev)
    need = ea.decode_workspace_size(w.B, w.Hq, w.Hkv, w.Nq, w.Nk, w.d, 0)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def call():
        ea.attn_fwd_decode(qd, kd, vd, causal=w.causal, scale=w.scale, out=out, lse=lse, workspace=ws,
                           stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            call()
    torch.cuda.synchronize(dev)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    with torch.cuda.stream(stream):
        for i in range(steps):
            flush_l2(flush)
            starts[i].record(stream)
            call()
            ends[i].record(stream)
    torch.cuda.synchronize(dev)
    return sum(a.elapsed_time(b) for a, b in zip(starts, ends)) / 1e3 / steps


def measure_bwd(ea, w: Workload, dev, steps: int, warmup: int, seed_offset: int = 0):
    """Device time per attn_bwd call (its three kernels) on workload w, with O and LSE
    from attn_fwd computed once beforehand; per-call CUDA events, L2 flushed between
    calls."""
    import torch
    from exact_self_attention_fwd_b300.inputs import make_dout
    q, k, v = make_qkv(w.B, w.Hq, w.Hkv, w.N, w.d, w.seed + seed_offset, w.q_head0_scale)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    dod = make_dout(w.B, w.Hq, w.N, w.d, w.seed + 100 + seed_offset).to(dev)
    stream = torch.cuda.Stream(dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    with torch.cuda.stream(stream):
        out, lse = ea.attn_fwd(qd, kd, vd, causal=w.causal, window=w.window, scale=w.scale, stream=stream)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    ws = torch.empty(ea.bwd_workspace_size(w.B, w.Hq, w.N, w.d), dtype=torch.uint8, device=dev)

    def call():
        ea.attn_bwd(qd, kd, vd, out, lse, dod, causal=w.causal, window=w.window, scale=w.scale,
                    dq=dq, dk=dk, dv=dv, workspace=ws, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(warmup):
            call()
    torch.cuda.synchronize(dev)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    with torch.cuda.stream(stream):
        for i in range(steps):
            flush_l2(flush)
            starts[i].record(stream)
            call()
            ends[i].record(stream)
    torch.cuda.synchronize(dev)
    return sum(a.elapsed_time(b) for a, b in zip(starts, ends)) / 1e3 / steps


def measure_fp8(ea, w: Workload, dev, steps: int, warmup: int, seed_offset: int = 0):
    """Device time per call of (a) attn_fwd_fp8 on pre-quantised operands, (b) the block
    quantisation of Q, K and V (three attn_quantize_e4m3 calls) and (c) the same with
    incoherent processing of Q and K (attn_quantize_e4m3_hadamard), per-call CUDA events
    with L2 flushed between calls."""
    import torch
    q, k, v = make_qkv(w.B, w.Hq, w.Hkv, w.N, w.d, w.seed + seed_offset, w.q_head0_scale)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    stream = torch.cuda.Stream(dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    with torch.cuda.stream(stream):
        (q8, qs), (k8, ks), (v8, vs) = (ea.quantize_e4m3(t, stream=stream) for t in (qd, kd, vd))
    out = torch.empty_like(qd)
    lse = torch.empty((w.B, w.Hq, w.N), dtype=torch.float32, device=dev)

    def attn():
        ea.attn_fwd_fp8(q8, k8, v8, qs, ks, vs, causal=w.causal, window=w.window, scale=w.scale, out=out,
                        lse=lse, stream=stream)

    def quant():
        for t in (qd, kd, vd):
            ea.quantize_e4m3(t, stream=stream)

    from exact_self_attention_fwd_b300.inputs import make_signs
    signs = make_signs(w.d, w.seed + 1) if w.d == 128 else None

    def quant_hadamard():
        # incoherent processing of Q and K, plain block quantisation of V
        ea.quantize_e4m3_hadamard(qd, signs, stream=stream)
        ea.quantize_e4m3_hadamard(kd, signs, stream=stream)
        ea.quantize_e4m3(vd, stream=stream)

    res = []
    for fn in (attn, quant, quant_hadamard):
        with torch.cuda.stream(stream):
            for _ in range(warmup):
                fn()
        torch.cuda.synchronize(dev)
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        with torch.cuda.stream(stream):
            for i in range(steps):
                flush_l2(flush)
                starts[i].record(stream)
                fn()
                ends[i].record(stream)
        torch.cuda.synchronize(dev)
        res.append(sum(a.elapsed_time(b) for a, b in zip(starts, ends)) / 1e3 / steps)
    return res[0], res[1], res[2]


def run_decode(args, w: DecodeWorkload):
    """One JSON line for a decode-shaped workload (one GPU; HBM roofline)."""
    import torch

    import exact_self_attention_fwd_b300 as ea
    world, rank, local = dist_env()
    dist = init_dist(world)
    if not torch.cuda.is_available():
        raise RuntimeError("no CUDA device: this benchmark times the CUDA library only")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    ea.load()
    sampler = ClockSampler(nvsmi_index(local), os.path.join(args.out_dir, f"clocks_rank{rank}.csv"))
    time.sleep(0.6)
    barrier(dist)
    t0 = time.time()
    t_call = measure_decode(ea, w, dev, args.steps, args.warmup, seed_offset=rank)
    barrier(dist)
    t1 = time.time()
    time.sleep(0.25)
    sampler.stop()
    if ea.device_error() != ea.ATTN_OK:
        raise RuntimeError("kernel wait timed out")
    t_max = max_over_ranks(dist, t_call)
    splits_ws = ea.decode_workspace_size(w.B, w.Hq, w.Hkv, w.Nq, w.Nk, w.d, 0)
    if rank == 0:
        peaks, peak_src = load_peaks()
        gbs = decode_hbm_bytes(w) / t_call / 1e9
        peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
        line = {
            "metric": "attention fwd TFLOP/s (unmasked FLOPs)", "value": decode_flops(w) * world / t_max / 1e12,
            "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": t_max * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic (seeded N(0,1) rounded to bf16)",
            "config": {"workload": w.name, "shape": w.note, "entry": "attn_fwd_decode",
                       "l2": "256 MiB buffer written then read before every call; per-call CUDA events exclude it",
                       "hbm_mb_per_step": decode_hbm_bytes(w) / 1e6},
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                         "traffic": recorded_traffic(w.name),
                         "peak_source": f"{peak_src} (MEASURED_PEAKS.json)" if peak_src == "measured" else "fallback",
                         "kernel": f"attn_fwd_kernel<{w.d}, decode>"},
            "cpu_baseline": None, "e2e": None,
            "gpu_launches": args.steps * (2 if splits_ws > 0 else 1),
            "clocks": sampler.summary(t0, t1),
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def run_ours(args, w: Workload):
    import torch

    import exact_self_attention_fwd_b300 as ea

    world, rank, local = dist_env()
    dist = init_dist(world)

    # CPU baseline first (before any GPU work), rank 0, N = 1 only
    cpu = None
    if rank == 0 and world == 1 and args.cpu_seconds > 0:
        val, cores, sample = oracle_sample(w, args.cpu_seconds, seed=7)
        cpu = {"value": val, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample}

    if not torch.cuda.is_available():
        raise RuntimeError("no CUDA device: this benchmark times the CUDA library only")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    ea.load()

    q, k, v = make_qkv(w.B, w.Hq, w.Hkv, w.N, w.d, w.seed + rank, w.q_head0_scale)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    out = torch.empty_like(qd)
    lse = torch.empty((w.B, w.Hq, w.N), dtype=torch.float32, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(dev)
    F = flops(w)

    def call():
        ea.attn_fwd(qd, kd, vd, causal=w.causal, window=w.window, scale=w.scale, out=out, lse=lse,
                    stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            flush_l2(flush)
            call()
    torch.cuda.synchronize(dev)
    if ea.device_error() != ea.ATTN_OK:
        raise RuntimeError("kernel wait timed out during warm-up")

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    sampler = ClockSampler(nvsmi_index(local), os.path.join(args.out_dir, f"clocks_rank{rank}.csv"))
    time.sleep(0.6)  # let nvidia-smi start sampling
    barrier(dist)
    torch.cuda.synchronize(dev)
    t0 = time.time()
    with torch.cuda.stream(stream):
        for i in range(args.steps):
            flush_l2(flush)
            starts[i].record(stream)
            call()
            ends[i].record(stream)
    torch.cuda.synchronize(dev)
    barrier(dist)
    t1 = time.time()
    time.sleep(0.25)
    sampler.stop()
    if ea.device_error() != ea.ATTN_OK:
        raise RuntimeError("kernel wait timed out in the timed region")
    per = [s.elapsed_time(e) for s, e in zip(starts, ends)]  # ms
    local_total = sum(per) / 1e3
    total = max_over_ranks(dist, local_total)
    value = F * world * args.steps / total / 1e12
    ms_step = 1e3 * total / args.steps
    srt = sorted(per)
    cut = int(len(srt) * 0.15)
    mid = srt[cut:len(srt) - cut] or srt
    clocks = sampler.summary(t0, t1)

    # end to end through the host-buffer entry point: pinned host inputs, H2D copies,
    # the kernel, D2H copies of O and LSE, all inside the timed region
    hq, hk, hv = q.pin_memory(), k.pin_memory(), v.pin_memory()
    ho = torch.empty_like(q).pin_memory()
    hl = torch.empty((w.B, w.Hq, w.N), dtype=torch.float32).pin_memory()
    e2e_steps = max(3, min(args.steps, 20))
    for _ in range(2):
        ea.attn_fwd_host(hq, hk, hv, ho, hl, qd, kd, vd, out, lse, causal=w.causal, window=w.window,
                         scale=w.scale, stream=stream)
    torch.cuda.synchronize(dev)
    es, ee = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist)
    torch.cuda.synchronize(dev)
    es.record(stream)
    for _ in range(e2e_steps):
        ea.attn_fwd_host(hq, hk, hv, ho, hl, qd, kd, vd, out, lse, causal=w.causal, window=w.window,
                         scale=w.scale, stream=stream)
    ee.record(stream)
    torch.cuda.synchronize(dev)
    barrier(dist)
    e2e_t = max_over_ranks(dist, es.elapsed_time(ee) / 1e3)
    h2d = hq.numel() * 2 + hk.numel() * 2 + hv.numel() * 2
    d2h = ho.numel() * 2 + hl.numel() * 4

    # every workload of the suite, measured the same way (short runs, reported beside
    # the headline; their launches are not counted in gpu_launches)
    summary = {}
    if args.summary_steps > 0:
        peaks, _ = load_peaks()
        for name, ww in WORKLOADS.items():
            t_call, how = measure_workload(ea, ww, dev, args.summary_steps, 5, seed_offset=rank)
            r = roofline_of(ww, t_call, peaks)
            summary[name] = {"tflops": flops(ww) / t_call / 1e12, "us_per_call": t_call * 1e6,
                             "gbs": hbm_bytes(ww) / t_call / 1e9, "bound": r["bound"],
                             "frac": r["frac"], "timing": how}
            if name in ("vit_base", "gpt2_small"):
                # the short-sequence workloads are also reported without the flush
                t_nf, _ = measure_workload(ea, ww, dev, args.summary_steps, 5, seed_offset=rank, flush=False)
                summary[name].update({"us_per_call_no_flush": t_nf * 1e6,
                                      "tflops_no_flush": flops(ww) / t_nf / 1e12,
                                      "gbs_no_flush": hbm_bytes(ww) / t_nf / 1e9})
        fw = WORKLOADS["gqa_8k"]
        t_attn, t_quant, t_quant_h = measure_fp8(ea, fw, dev, args.summary_steps, 5, seed_offset=rank)
        fp8_peak = 2.0 * float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
        qbytes = (fw.B * fw.Hq + 2 * fw.B * fw.Hkv) * fw.N * fw.d * 3  # read bf16, write e4m3
        summary["gqa_8k_fp8"] = {
            "tflops": flops(fw) / t_attn / 1e12, "us_per_call": t_attn * 1e6, "bound": "tensor",
            "frac": flops(fw) / t_attn / 1e12 / fp8_peak,
            "peak_note": "fp8 peak = 2 x measured bf16 burst peak (nominal dense ratio)",
            "quantize_us": t_quant * 1e6, "quantize_gbs": qbytes / t_quant / 1e9,
            "quantize_hadamard_us": t_quant_h * 1e6, "quantize_hadamard_gbs": qbytes / t_quant_h / 1e9,
            "timing": "per-call CUDA events, L2 flushed between calls",
            "entry": ("attn_fwd_fp8 (e4m3 Q, K, V with 128-row block scales); attn_quantize_e4m3 and "
                      "attn_quantize_e4m3_hadamard (incoherent processing of Q and K) timed apart")}
        for name in ("gpt2_small", "gqa_8k"):
            bw = WORKLOADS[name]
            t_bwd = measure_bwd(ea, bw, dev, args.summary_steps, 3, seed_offset=rank)
            tf = bwd_flops(bw) / t_bwd / 1e12
            summary[name + "_bwd"] = {
                "tflops": tf, "us_per_call": t_bwd * 1e6, "bound": "tensor",
                "frac": tf / float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])),
                "flops_note": "5 products of d MACs per visible pair (2.5 x the forward)",
                "timing": "per-call CUDA events, L2 flushed between calls",
                "entry": "attn_bwd (row-term preprocess + dK/dV kernel + dQ kernel)"}
        for name, dw in DECODE_WORKLOADS.items():
            t_call = measure_decode(ea, dw, dev, args.summary_steps, 5, seed_offset=rank)
            gbs = decode_hbm_bytes(dw) / t_call / 1e9
            summary[name] = {"tflops": decode_flops(dw) / t_call / 1e12, "us_per_call": t_call * 1e6,
                             "gbs": gbs, "bound": "hbm",
                             "frac": gbs / float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])),
                             "timing": "per-call CUDA events, L2 flushed between calls",
                             "entry": "attn_fwd_decode (split key sequence + merge kernel)",
                             "shape": dw.note}

    if rank == 0:
        peaks, peak_src = load_peaks()
        avg_s = local_total / args.steps
        roof = roofline_of(w, avg_s, peaks)
        roof["traffic"] = recorded_traffic(w.name)
        roof["peak_source"] = f"{peak_src} (MEASURED_PEAKS.json burst)" if peak_src == "measured" else "fallback"
        roof["kernel"] = f"attn_fwd_kernel<{w.d}>"
        line = {
            "metric": "attention fwd TFLOP/s (unmasked FLOPs)", "value": value, "unit": "TFLOP/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) rounded to bf16)",
            "config": {"workload": w.name, "shape": w.note, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv,
                       "N": w.N, "d": w.d, "causal": w.causal, "window": w.window,
                       "l2": "256 MiB buffer written then read before every call; per-call CUDA events exclude it",
                       "parallelism": f"replica per GPU x{world}",
                       "gflop_per_step": F / 1e9, "hbm_mb_per_step": hbm_bytes(w) / 1e6},
            "roofline": roof,
            "cpu_baseline": cpu,
            "e2e": {"value": F * world * e2e_steps / e2e_t / 1e12, "unit": "TFLOP/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "entry": "attn_fwd_host (pinned host buffers)"},
            "gpu_launches": args.steps,
            "clocks": clocks,
            "stats_ms": {"mean": statistics.mean(per), "median": statistics.median(per),
                         "min": min(per), "trimmed_mean_70": statistics.mean(mid)},
            "workloads": summary,
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def run_bwd(args, w: Workload):
    """The backward pass as the timed step (one GPU): attn_bwd on the workload with O and
    LSE from one attn_fwd call made beforehand, per-call CUDA events, L2 flushed between
    calls. Used to measure and profile the backward kernels on their own."""
    import torch

    import exact_self_attention_fwd_b300 as ea
    world, _, local = dist_env()
    if world != 1:
        raise RuntimeError("--pass bwd runs on one GPU")
    if not torch.cuda.is_available():
        raise RuntimeError("no CUDA device: this benchmark times the CUDA library only")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    ea.load()
    t = measure_bwd(ea, w, dev, args.steps, args.warmup)
    if ea.device_error() != ea.ATTN_OK:
        raise RuntimeError("kernel wait timed out")
    peaks, peak_src = load_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    tf = bwd_flops(w) / t / 1e12
    line = {
        "metric": "attention bwd TFLOP/s (10 d FLOP per visible pair, 2.5 x the forward)", "value": tf,
        "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) rounded to bf16)",
        "config": {"workload": w.name, "pass": "bwd", "shape": w.note,
                   "l2": "256 MiB buffer written then read before every call; per-call CUDA events exclude it"},
        "roofline": {"bound": "tensor", "achieved": tf, "peak": peak, "unit": "TFLOP/s", "frac": tf / peak,
                     "traffic": None, "peak_source": peak_src,
                     "kernel": f"bwd_preprocess_kernel<{w.d}> + attn_bwd_kernel<{w.d}, 0> + attn_bwd_kernel<{w.d}, 1>"},
        "gpu_launches": 3 * args.steps,
    }
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS) + sorted(DECODE_WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--pass", dest="which", default="fwd", choices=["fwd", "bwd"],
                    help="bwd: time attn_bwd on the workload instead (one GPU, no reference arm)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="seconds of oracle work for the cpu_baseline field (0 = skip)")
    ap.add_argument("--ref-seconds", type=float, default=90.0,
                    help="total oracle seconds for --impl reference")
    ap.add_argument("--summary-steps", type=int, default=100,
                    help="calls per workload for the all-workload summary (0 = skip)")
    ap.add_argument("--out-dir", default=os.path.join(ROOT, "bench_out"),
                    help="where the nvidia-smi clock samples are written")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    os.makedirs(args.out_dir, exist_ok=True)
    if args.workload in DECODE_WORKLOADS:
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the oracle arm times the prefill workloads"}))
            return 0
        return run_decode(args, DECODE_WORKLOADS[args.workload])
    w = WORKLOADS[args.workload]
    if args.which == "bwd":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable": "the oracle arm times the forward"}))
            return 0
        return run_bwd(args, w)
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
