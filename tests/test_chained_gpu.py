"""Dependent calls queued back to back on one stream.

Every kernel of the library is launched as a programmatic dependent of the kernel before
it on the stream: its prologue may run while that kernel finishes, and it waits for it
(griddepcontrol.wait) before its first memory access. These tests chain calls whose
inputs are the previous call's outputs, with no synchronisation in between (also inside
a CUDA graph), and require the results to equal, bit for bit, the same chain run with a
device synchronisation after every call.
"""
from __future__ import annotations

import pytest
import torch

import exact_self_attention_fwd_b300 as ea
from exact_self_attention_fwd_b300.inputs import make_dout, make_qkv, make_qkv_decode

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
STEPS = 6


def _chain(q, k, v, causal, window, sync):
    """q_{i+1} = attn(q_i, k, v): each call reads the output the previous one wrote."""
    outs = []
    x = q
    for _ in range(STEPS):
        o, lse = ea.attn_fwd(x, k, v, causal=causal, window=window)
        outs.append((o, lse))
        if sync:
            torch.cuda.synchronize()
        x = o
    torch.cuda.synchronize()
    return outs


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal,W", [(True, 0), (False, 0), (True, 200)])
def test_forward_chain_matches_synchronised(d, causal, W):
    q, k, v = (t.to(DEV) for t in make_qkv(2, 8, 2, 700, d, 8100 + d))
    ref = _chain(q, k, v, causal, W, sync=True)
    got = _chain(q, k, v, causal, W, sync=False)
    for (o_r, l_r), (o_g, l_g) in zip(ref, got):
        assert torch.equal(o_r, o_g) and torch.equal(l_r, l_g)
    assert ea.device_error() == ea.ATTN_OK


def test_forward_chain_in_a_cuda_graph():
    q, k, v = (t.to(DEV) for t in make_qkv(1, 4, 4, 300, 128, 8200))
    ref = _chain(q, k, v, True, 0, sync=True)
    x_in = q.clone()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        ea.attn_fwd(x_in, k, v, causal=True)  # warm-up outside the capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        outs = []
        with torch.cuda.graph(g, stream=s):
            x = x_in
            for _ in range(STEPS):
                o, lse = ea.attn_fwd(x, k, v, causal=True)
                outs.append((o, lse))
                x = o
        g.replay()
    torch.cuda.synchronize()
    for (o_r, l_r), (o_g, l_g) in zip(ref, outs):
        assert torch.equal(o_r, o_g) and torch.equal(l_r, l_g)
    assert ea.device_error() == ea.ATTN_OK


@pytest.mark.parametrize("splits", [1, 3])
def test_decode_chain_matches_synchronised(splits):
    """The split kernel and its merge kernel, call after call: q_{i+1} = o_i."""
    q, k, v = (t.to(DEV) for t in make_qkv_decode(4, 32, 8, 2, 3000, 128, 8300 + splits))

    def run(sync):
        outs, x = [], q
        for _ in range(STEPS):
            o, lse = ea.attn_fwd_decode(x, k, v, causal=True, splits=splits)
            outs.append((o, lse))
            if sync:
                torch.cuda.synchronize()
            x = o
        torch.cuda.synchronize()
        return outs

    for (o_r, l_r), (o_g, l_g) in zip(run(True), run(False)):
        assert torch.equal(o_r, o_g) and torch.equal(l_r, l_g)
    assert ea.device_error() == ea.ATTN_OK


@pytest.mark.parametrize("d", [64, 128])
def test_forward_then_backward_chain(d):
    """Forward, backward (row-term kernel, dK/dV kernel, dQ kernel) and a forward on the
    gradients, queued without synchronisation."""
    q, k, v = (t.to(DEV) for t in make_qkv(2, 8, 2, 520, d, 8400 + d))
    do = make_dout(2, 8, 520, d, 8401 + d).to(DEV)

    def run(sync):
        o, lse = ea.attn_fwd(q, k, v, causal=True)
        if sync:
            torch.cuda.synchronize()
        dq, dk, dv = ea.attn_bwd(q, k, v, o, lse, do, causal=True)
        if sync:
            torch.cuda.synchronize()
        o2, lse2 = ea.attn_fwd(dq, dk, dv, causal=True)
        torch.cuda.synchronize()
        return o, lse, dq, dk, dv, o2, lse2

    for a, b in zip(run(True), run(False)):
        assert torch.equal(a, b)
    assert ea.device_error() == ea.ATTN_OK
