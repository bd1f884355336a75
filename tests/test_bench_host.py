"""Host-side logic of bench.py, on CPU: FLOP and byte accounting, the clock-sample
parser, the traffic record, the reference (oracle) arm, and the multi-rank timing
reduction over two gloo ranks."""
from __future__ import annotations

import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from exact_self_attention_fwd_b300.inputs import WORKLOADS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def brute_pairs(N, causal, window):
    i = np.arange(N)[:, None]
    j = np.arange(N)[None, :]
    vis = np.ones((N, N), dtype=bool)
    if causal:
        vis &= j <= i
    if window:
        vis &= (i - j) < window
    return int(vis.sum())


@pytest.mark.parametrize("N", [1, 2, 7, 128, 197, 300])
@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 1), (True, 5), (True, 128),
                                           (True, 299), (True, 300), (True, 10000)])
def test_visible_pairs_brute_force(N, causal, window):
    assert bench.visible_pairs(N, causal, window) == brute_pairs(N, causal, window)


def test_workload_accounting():
    # pairs per (batch, head): N^2 bidirectional, N(N+1)/2 causal, and for the window
    # W(W+1)/2 + (N-W)W; FLOPs count 4*d per visible pair (two products of d MACs)
    expect = {"tiny": 128 * 128, "vit_base": 197 * 197, "gpt2_small": 1024 * 1025 // 2,
              "gqa_8k": 8192 * 8193 // 2, "swa_16k": 1024 * 1025 // 2 + (16384 - 1024) * 1024}
    for name, w in WORKLOADS.items():
        assert bench.visible_pairs(w.N, w.causal, w.window) == expect[name]
        assert bench.flops(w) == 4 * w.B * w.Hq * expect[name] * w.d
        assert bench.bwd_flops(w) * 2 == bench.flops(w) * 5
    w = WORKLOADS["gqa_8k"]
    assert bench.hbm_bytes(w) == (2 * 32 * 8192 * 128 * 2) * 2 + 2 * (2 * 8 * 8192 * 128 * 2) + 2 * 32 * 8192 * 4


def test_clock_summary_parses_nvidia_smi_csv(tmp_path):
    path = tmp_path / "clocks.csv"
    path.write_text(
        "timestamp, index, clocks.current.sm [MHz], clocks.max.sm [MHz], power.draw [W], "
        "clocks_event_reasons.active, clocks_event_reasons.hw_slowdown, "
        "clocks_event_reasons.hw_thermal_slowdown, clocks_event_reasons.sw_thermal_slowdown, "
        "clocks_event_reasons.sw_power_cap\n"
        "2026/12/02 15:44:00.100, 0, 2032, 2032, 500.0, 0x0, Not Active, Not Active, Not Active, Not Active\n"
        "2026/12/02 15:44:00.300, 0, 1900, 2032, 1090.0, 0x4, Not Active, Not Active, Not Active, Active\n"
        "2026/12/02 15:44:00.500, 0, 1950, 2032, 1095.0, 0x4, Not Active, Not Active, Not Active, Active\n"
        "2026/12/02 15:44:09.000, 0, 1000, 2032, 100.0, 0x0, Active, Not Active, Not Active, Not Active\n")
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.path = str(path)
    s.proc = object()
    import time
    t0 = time.mktime(time.strptime("2026/12/02 15:44:00", "%Y/%m/%d %H:%M:%S")) + 0.2
    out = s.summary(t0, t0 + 0.4)
    assert out["samples_in_region"] == 2
    assert out["sm_mhz"] == pytest.approx(1925.0)
    assert out["sm_max_mhz"] == 2032.0
    assert out["reasons"] == ["sw_power_cap"]   # the hw_slowdown sample lies outside the region


def test_recorded_traffic_requires_current_kernel(tmp_path, monkeypatch):
    f = tmp_path / "traffic.txt"
    f.write_text(f"# workload bytes sha note\ngqa_8k 123456789 {bench.kernel_sha()} note\n"
                 "swa_16k 5 0000000000000000 stale\n")
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.recorded_traffic("gqa_8k") == 123456789
    assert bench.recorded_traffic("swa_16k") is None     # taken on another kernel
    assert bench.recorded_traffic("vit_base") is None


def test_reference_arm_prints_one_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "tiny", "--steps", "2", "--warmup", "3", "--ref-seconds", "2"],
                         capture_output=True, text=True, timeout=300, check=True).stdout
    lines = [l for l in out.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["config"]["workload"] == "tiny"


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    d = bench.init_dist(world)
    bench.barrier(d)
    got = bench.max_over_ranks(d, 1.0 + rank * 0.5)
    q.put((rank, got))
    d.destroy_process_group()


def test_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + (os.getpid() % 1000)
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == {0: 1.5, 1: 1.5}


def test_decode_accounting():
    from exact_self_attention_fwd_b300.inputs import DecodeWorkload
    w = DecodeWorkload("t", 2, 8, 2, 3, 10, 64, True, 0)
    # positions 7, 8, 9 see 8, 9, 10 keys
    assert bench.decode_flops(w) == 4 * 2 * 8 * (8 + 9 + 10) * 64
    wb = DecodeWorkload("t", 2, 8, 2, 3, 10, 64, False, 0)
    assert bench.decode_flops(wb) == 4 * 2 * 8 * 30 * 64
    assert bench.decode_hbm_bytes(w) == 2 * (2 * 8 * 3 * 64 * 2) + 2 * (2 * 2 * 10 * 64 * 2) + 2 * 8 * 3 * 4


def test_kernel_sha_covers_the_forward_kernel_only(tmp_path, monkeypatch):
    # the hash follows the forward kernel's device code, its launch function and ptx.cuh,
    # and ignores the rest of the translation unit (quantisers, decode merge, backward)
    for rel in bench.KERNEL_SOURCES:
        dst = tmp_path / rel
        dst.parent.mkdir(parents=True, exist_ok=True)
        dst.write_bytes(open(os.path.join(ROOT, rel), "rb").read())
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    base = bench.kernel_sha()
    assert base == bench.kernel_sha() and len(base) == 16
    cu = next(tmp_path / rel for rel in bench.KERNEL_SOURCES if rel.endswith("attn_fwd.cu"))
    src = cu.read_text()
    assert src.count("// Block quantisation to e4m3") == 1 and src.count("int launch(const void *q") == 1
    # an edit to a later kernel (the e4m3 quantiser) leaves the hash alone
    cu.write_text(src.replace("// Block quantisation to e4m3", "// Block quantisation to e4m3\n// x", 1))
    assert bench.kernel_sha() == base
    # an edit inside the forward kernel changes it
    cu.write_text(src.replace("attn_fwd_kernel(", "attn_fwd_kernel (", 1))
    assert bench.kernel_sha() != base
    cu.write_text(src)
    assert bench.kernel_sha() == base


def test_roofline_labels():
    # the one-tile workload is launch-latency bound: its figure is microseconds per
    # call, with no fraction of a throughput peak; the others report a fraction
    import bench
    from exact_self_attention_fwd_b300.inputs import WORKLOADS
    peaks = {"hbm_gbs": 6000.0, "bf16_tflops": 1700.0, "bf16_tflops_sustained": 1400.0}
    r = bench.roofline_of(WORKLOADS["tiny"], 5e-6, peaks)
    assert r["bound"] == "latency" and r["frac"] is None and abs(r["achieved"] - 5.0) < 1e-9
    assert bench.roofline_of(WORKLOADS["vit_base"], 1e-4, peaks)["bound"] == "hbm"
    r = bench.roofline_of(WORKLOADS["gqa_8k"], 7e-4, peaks)
    assert r["bound"] == "tensor" and 0 < r["frac"] < 1.5
