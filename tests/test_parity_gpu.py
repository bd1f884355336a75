"""The CUDA path (through the C ABI) against the fp64 oracle, element by element."""
from __future__ import annotations

import json
import math

import numpy as np
import pytest
import torch

import oracle
import exact_self_attention_fwd_b300 as ea
from exact_self_attention_fwd_b300.inputs import WORKLOADS, make_qkv, make_workload
from parity import compare

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def run_gpu(q, k, v, causal, window, scale):
    out, lse = ea.attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal, window=window, scale=scale)
    torch.cuda.synchronize()
    assert ea.device_error() == ea.ATTN_OK
    return out, lse


def check_full(B, Hq, Hkv, N, d, causal, window, seed, scale=None, q_head0_scale=1.0):
    q, k, v = make_qkv(B, Hq, Hkv, N, d, seed, q_head0_scale)
    scale = scale or 1.0 / math.sqrt(d)
    out, lse = run_gpu(q, k, v, causal, window, scale)
    o_ref, lse_ref = oracle.attn_ref(q, k, v, causal=causal, window=window, scale=scale)
    return compare(out, lse, o_ref, lse_ref, f"B{B} Hq{Hq} Hkv{Hkv} N{N} d{d} c{causal} W{window}")


# ------------------------------------------------------------ sequence lengths and tails
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 2, 17, 127, 128, 129, 197, 255, 256, 257, 300, 513])
def test_lengths(N, d, causal):
    check_full(2, 3, 3, N, d, causal, 0, seed=1000 + N + d + int(causal))


# ------------------------------------------------------------ grouped-query heads
@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("causal", [False, True])
def test_gqa(G, causal):
    check_full(2, 8, 8 // G, 300, 128, causal, 0, seed=2000 + G)
    check_full(1, 8, 8 // G, 260, 64, causal, 0, seed=2100 + G)


# ------------------------------------------------------------ sliding window
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("W", [1, 2, 100, 127, 128, 129, 255, 256, 300, 599, 600, 1000])
def test_window(W, d):
    check_full(1, 2, 1, 600, d, True, W, seed=3000 + W)


def test_window_ge_n_equals_causal():
    q, k, v = make_qkv(1, 4, 2, 333, 128, 77)
    a = run_gpu(q, k, v, True, 0, 0.088)
    b = run_gpu(q, k, v, True, 333, 0.088)
    c = run_gpu(q, k, v, True, 5000, 0.088)
    assert torch.equal(a[0], b[0]) and torch.equal(a[0], c[0])
    assert torch.equal(a[1], b[1]) and torch.equal(a[1], c[1])


# ------------------------------------------------------------ softmax range
@pytest.mark.parametrize("mult", [0.0, 4.0, 16.0])
def test_sharp_and_flat_softmax(mult):
    g = torch.Generator().manual_seed(5)
    q = (mult * torch.randn(1, 2, 384, 64, generator=g)).bfloat16()
    k = torch.randn(1, 2, 384, 64, generator=g).bfloat16()
    v = torch.randn(1, 2, 384, 64, generator=g).bfloat16()
    for causal in (False, True):
        out, lse = run_gpu(q, k, v, causal, 0, 0.125)
        o_ref, lse_ref = oracle.attn_ref(q, k, v, causal=causal, scale=0.125)
        compare(out, lse, o_ref, lse_ref, f"mult {mult} causal {causal}")


def test_many_units_per_cta():
    # more work units than SMs: exercises the persistent loop and barrier phases
    check_full(4, 40, 8, 520, 64, True, 0, seed=6)
    check_full(3, 64, 16, 260, 128, False, 0, seed=7)


# ------------------------------------------------------------ the five workloads, every row
@pytest.mark.parametrize("name", ["tiny", "vit_base", "gpt2_small", "gqa_8k", "swa_16k"])
def test_workload_every_row(name):
    """Each benchmark workload at its full size, in the launch configuration the
    benchmark times, every output element against the oracle: the bf16 output under the
    stated bar (elements excused only by the bf16 format floor are counted), and the
    fp32 output of the same kernel (attn_fwd_o32) under the plain bar, max <= 1e-2 and
    mean <= 1e-3 with no allowance. The bf16 O must be the fp32 O rounded to nearest
    even, bit for bit, and the two LSEs identical."""
    w = WORKLOADS[name]
    q, k, v = make_workload(w)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    out, lse = ea.attn_fwd(qd, kd, vd, causal=w.causal, window=w.window, scale=w.scale)
    o32, lse32 = ea.attn_fwd(qd, kd, vd, causal=w.causal, window=w.window, scale=w.scale, out_fp32=True)
    torch.cuda.synchronize()
    assert ea.device_error() == ea.ATTN_OK
    assert torch.equal(out, o32.to(torch.bfloat16)) and torch.equal(lse, lse32)
    o_ref, lse_ref = oracle.attn_ref(q, k, v, causal=w.causal, window=w.window, scale=w.scale)
    stats = compare(out, lse, o_ref, lse_ref, w.name)
    strict = compare(o32, lse32, o_ref, lse_ref, w.name + " fp32 output", strict=True)
    print(json.dumps({"workload": name, "bf16_output": stats, "fp32_output": strict}))
    # properties of every row: a convex combination of V rows, and lse_i >= s_ii (the
    # diagonal is always visible under these masks)
    vmax = v.float().abs().amax().item()
    assert o32.abs().amax().item() <= vmax * (1 + 2 ** -7)
    kd_rep = kd.float().repeat_interleave(w.group, dim=1)
    s_ii = (qd.float() * kd_rep).sum(-1) * w.scale
    assert bool((lse >= s_ii - 1e-3 * s_ii.abs().clamp(min=1)).all())


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal,W,N", [(False, 0, 1), (False, 0, 129), (True, 0, 300), (True, 100, 513),
                                        (False, 77, 260)])
def test_fp32_output_plain_bar(N, d, causal, W):
    """attn_fwd_o32 on ragged lengths and masks: the plain bar, and bf16 O = rne(fp32 O)."""
    q, k, v = make_qkv(2, 4, 2, N, d, 6000 + N + d + W)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    scale = 1.0 / math.sqrt(d)
    o32, lse32 = ea.attn_fwd(qd, kd, vd, causal=causal, window=W, scale=scale, out_fp32=True)
    out, lse = ea.attn_fwd(qd, kd, vd, causal=causal, window=W, scale=scale)
    torch.cuda.synchronize()
    assert ea.device_error() == ea.ATTN_OK
    assert torch.equal(out, o32.to(torch.bfloat16)) and torch.equal(lse, lse32)
    o_ref, lse_ref = oracle.attn_ref(q, k, v, causal=causal, window=W, scale=scale)
    compare(o32, lse32, o_ref, lse_ref, f"fp32 N{N} d{d} c{causal} W{W}", strict=True)


def test_fp32_output_with_padding():
    key_len = [0, 1, 129, 300]
    q, k, v = make_qkv(4, 4, 2, 300, 128, 6100)
    kl = torch.tensor(key_len, dtype=torch.int32, device=DEV)
    o32, lse32 = ea.attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=True, key_len=kl, out_fp32=True)
    out, lse = ea.attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=True, key_len=kl)
    torch.cuda.synchronize()
    assert torch.equal(out, o32.to(torch.bfloat16)) and torch.equal(lse, lse32)
    o_ref, lse_ref = oracle.attn_ref(q, k, v, causal=True, scale=128 ** -0.5, key_len=key_len)
    live = np.isfinite(lse_ref)
    assert np.all(lse32.cpu().numpy()[~live] == -np.inf) and bool((o32.cpu().numpy()[~live] == 0).all())
    compare(o32[torch.from_numpy(live).to(DEV)], lse32[torch.from_numpy(live).to(DEV)], o_ref[live],
            lse_ref[live], "fp32 padded", strict=True)


# ------------------------------------------------------------ determinism, streams, host entry
def test_deterministic():
    q, k, v = make_qkv(2, 8, 2, 1000, 128, 8)
    a = run_gpu(q, k, v, True, 0, 0.09)
    b = run_gpu(q, k, v, True, 0, 0.09)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_side_stream_matches_default():
    q, k, v = make_qkv(1, 4, 4, 400, 64, 9)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    a = ea.attn_fwd(qd, kd, vd, causal=True)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        b = ea.attn_fwd(qd, kd, vd, causal=True, stream=s)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_host_entry_matches_device_entry():
    B, Hq, Hkv, N, d = 2, 8, 4, 300, 128
    q, k, v = make_qkv(B, Hq, Hkv, N, d, 10)
    ref = run_gpu(q, k, v, True, 64, 0.1)
    hq, hk, hv = q.pin_memory(), k.pin_memory(), v.pin_memory()
    ho = torch.empty_like(q).pin_memory()
    hl = torch.empty(B, Hq, N, dtype=torch.float32).pin_memory()
    dq, dk, dv = torch.empty_like(q, device=DEV), torch.empty_like(k, device=DEV), torch.empty_like(v, device=DEV)
    do = torch.empty_like(q, device=DEV)
    dl = torch.empty(B, Hq, N, dtype=torch.float32, device=DEV)
    ea.attn_fwd_host(hq, hk, hv, ho, hl, dq, dk, dv, do, dl, causal=True, window=64, scale=0.1)
    torch.cuda.synchronize()
    assert torch.equal(ho, ref[0].cpu()) and torch.equal(hl, ref[1].cpu())


def _host_call(q, k, v, causal, window, scale, stream=None, keep=None):
    """The copies are asynchronous: the pinned inputs must outlive them (until the
    stream is synchronised), so they are appended to `keep`, or to a module list."""
    B, Hq, N, d = q.shape
    hq, hk, hv = q.pin_memory(), k.pin_memory(), v.pin_memory()
    ho = torch.empty_like(q).pin_memory()
    hl = torch.empty(B, Hq, N, dtype=torch.float32).pin_memory()
    dq, dk, dv = torch.empty_like(q, device=DEV), torch.empty_like(k, device=DEV), torch.empty_like(v, device=DEV)
    do = torch.empty_like(q, device=DEV)
    dl = torch.empty(B, Hq, N, dtype=torch.float32, device=DEV)
    ea.attn_fwd_host(hq, hk, hv, ho, hl, dq, dk, dv, do, dl, causal=causal, window=window, scale=scale,
                     stream=stream)
    (_PINNED if keep is None else keep).extend([hq, hk, hv])
    return ho, hl, (dq, dk, dv, do, dl)


_PINNED = []


@pytest.mark.parametrize("B,Hq,Hkv,N,d", [(3, 10, 5, 260, 64), (1, 4, 1, 300, 128), (2, 16, 8, 129, 128)])
def test_host_entry_chunks(B, Hq, Hkv, N, d):
    # 15 groups over 8 chunks (uneven), a single group, 16 groups over 8 chunks: the
    # pipelined host entry gives the device entry's bits
    q, k, v = make_qkv(B, Hq, Hkv, N, d, 12 + B + Hkv)
    ref = run_gpu(q, k, v, True, 0, 0.1)
    ho, hl, _ = _host_call(q, k, v, True, 0, 0.1)
    torch.cuda.synchronize()
    assert torch.equal(ho, ref[0].cpu()) and torch.equal(hl, ref[1].cpu())


def test_host_entry_back_to_back_and_threads():
    # two calls in a row reusing the same device buffers, then two host threads at
    # once on two streams: every result equals its own device-entry result
    import threading
    cases = [make_qkv(2, 8, 2, 700, 128, 30 + i) for i in range(3)]
    refs = [run_gpu(q, k, v, True, 0, 0.09) for q, k, v in cases]
    q, k, v = cases[0]
    ho, hl, bufs = _host_call(q, k, v, True, 0, 0.09)
    q2, k2, v2 = cases[1]
    hq2, hk2, hv2 = q2.pin_memory(), k2.pin_memory(), v2.pin_memory()
    ho2 = torch.empty_like(q2).pin_memory()
    hl2 = torch.empty(2, 8, 700, dtype=torch.float32).pin_memory()
    ea.attn_fwd_host(hq2, hk2, hv2, ho2, hl2, *bufs, causal=True, window=0, scale=0.09)
    torch.cuda.synchronize()
    assert torch.equal(ho, refs[0][0].cpu()) and torch.equal(hl, refs[0][1].cpu())
    assert torch.equal(ho2, refs[1][0].cpu()) and torch.equal(hl2, refs[1][1].cpu())
    out = {}

    def worker(i):
        torch.cuda.set_device(0)
        st = torch.cuda.Stream()
        qq, kk, vv = cases[i]
        with torch.cuda.stream(st):
            out[i] = _host_call(qq, kk, vv, True, 0, 0.09, stream=st)[:2]
        st.synchronize()

    ts = [threading.Thread(target=worker, args=(i,)) for i in (1, 2)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    torch.cuda.synchronize()
    for i in (1, 2):
        assert torch.equal(out[i][0], refs[i][0].cpu()) and torch.equal(out[i][1], refs[i][1].cpu())


def test_output_buffers_untouched_outside_shape():
    # the kernel writes exactly B*Hq*N rows: a guard region after O and LSE stays intact
    q, k, v = make_qkv(1, 2, 2, 197, 64, 11)
    big_o = torch.full((2 * 197 * 64 + 4096,), 7.0, dtype=torch.bfloat16, device=DEV)
    big_l = torch.full((2 * 197 + 1024,), 7.0, dtype=torch.float32, device=DEV)
    o = big_o[: 2 * 197 * 64].view(1, 2, 197, 64)
    l = big_l[: 2 * 197].view(1, 2, 197)
    ea.attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), out=o, lse=l)
    torch.cuda.synchronize()
    assert bool((big_o[2 * 197 * 64:] == 7.0).all()) and bool((big_l[2 * 197:] == 7.0).all())


def test_bad_arguments_raise():
    q = torch.zeros(1, 3, 64, 64, dtype=torch.bfloat16, device=DEV)
    k = torch.zeros(1, 2, 64, 64, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(ea.AttnError) as e:
        ea.attn_fwd(q, k, k)
    assert e.value.code == ea.ATTN_ERR_SHAPE
    q = torch.zeros(1, 1, 64, 96, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(ea.AttnError) as e:
        ea.attn_fwd(q, q, q)
    assert e.value.code == ea.ATTN_ERR_UNSUPPORTED


# ------------------------------------------------------------ symmetric window and padding
def check_masked(B, Hq, Hkv, N, d, causal, window, seed, key_len=None, scale=None):
    q, k, v = make_qkv(B, Hq, Hkv, N, d, seed)
    scale = scale or 1.0 / math.sqrt(d)
    kl = None if key_len is None else torch.tensor(key_len, dtype=torch.int32, device=DEV)
    out, lse = ea.attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal, window=window, scale=scale,
                           key_len=kl)
    torch.cuda.synchronize()
    assert ea.device_error() == ea.ATTN_OK
    o_ref, lse_ref = oracle.attn_ref(q, k, v, causal=causal, window=window, scale=scale, key_len=key_len)
    dead = ~np.isfinite(lse_ref)           # rows with no visible key (padding)
    o_g = out.float().cpu().numpy()
    l_g = lse.cpu().numpy()
    assert np.all(l_g[dead] == -np.inf) and np.all(o_g[dead] == 0.0), "padded rows must be o=0, lse=-inf"
    live = ~dead
    label = f"B{B} Hq{Hq} Hkv{Hkv} N{N} d{d} c{causal} W{window} L{key_len}"
    return compare(out[torch.from_numpy(live).to(DEV)], lse[torch.from_numpy(live).to(DEV)],
                   o_ref[live], lse_ref[live], label)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("W", [1, 2, 64, 127, 128, 129, 200, 300, 599, 600, 10000])
def test_symmetric_window(W, d):
    check_masked(1, 2, 1, 600, d, False, W, seed=4000 + W)


@pytest.mark.parametrize("N,W", [(1, 1), (129, 5), (257, 128), (1000, 256)])
def test_symmetric_window_lengths(N, W):
    check_masked(2, 4, 2, N, 128, False, W, seed=4100 + N)
    check_masked(2, 4, 4, N, 64, False, W, seed=4200 + N)


@pytest.mark.parametrize("causal,W", [(False, 0), (True, 0), (True, 100), (False, 100)])
@pytest.mark.parametrize("d", [64, 128])
def test_padding(causal, W, d):
    # lengths: empty, one token, inside a tile, tile edges, full
    key_len = [0, 1, 77, 128, 129, 255, 256, 300, 513, 700]
    check_masked(len(key_len), 4, 2, 700, d, causal, W, seed=4300 + d + W, key_len=key_len)


def test_padding_full_length_equals_unpadded():
    q, k, v = make_qkv(2, 4, 4, 333, 64, 44)
    a = ea.attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=True)
    kl = torch.full((2,), 333, dtype=torch.int32, device=DEV)
    b = ea.attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=True, key_len=kl)
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_padding_many_units():
    rng = np.random.default_rng(5)
    key_len = [int(x) for x in rng.integers(0, 1025, size=24)]
    check_masked(24, 8, 2, 1024, 128, True, 0, seed=4400, key_len=key_len)
    check_masked(24, 8, 8, 1024, 64, False, 0, seed=4401, key_len=key_len)


# ------------------------------------------------------------ mask edges on 32-column chunks
# Edge tiles skip, warp by warp, the 32-column chunks inside every row's key interval and
# compare the rest element by element. These place the sequence end, the window's lower
# edge and the padding length exactly on chunk boundaries and one past them.
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [32, 33, 64, 96, 160, 192, 224, 225])
def test_sequence_end_on_chunk_boundaries(N, d, causal):
    check_full(1, 2, 1, N, d, causal, 0, seed=5000 + N + d + int(causal))


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("W", [32, 33, 96, 160, 224])
def test_window_edge_on_chunk_boundaries(W, d):
    check_full(1, 2, 1, 450, d, True, W, seed=5100 + W + d)
    check_masked(1, 2, 1, 450, d, False, W, seed=5200 + W + d)


@pytest.mark.parametrize("d", [64, 128])
def test_padding_on_chunk_boundaries(d):
    key_len = [32, 64, 96, 160, 192, 224, 31, 97]
    check_masked(len(key_len), 2, 1, 256, d, True, 0, seed=5300 + d, key_len=key_len)
    check_masked(len(key_len), 2, 1, 256, d, False, 0, seed=5400 + d, key_len=key_len)
