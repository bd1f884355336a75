"""The decode-shaped forward (queries at the end of a long key/value sequence, key
tiles split across CTAs and merged by log-sum-exp) through the C ABI, against the
fp64 oracle's decode shape, element by element."""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
import exact_self_attention_fwd_b300 as ea
from exact_self_attention_fwd_b300.inputs import make_qkv_decode
from parity import compare

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def run_decode(B, Hq, Hkv, Nq, Nk, d, causal, window, splits, seed):
    q, k, v = make_qkv_decode(B, Hq, Hkv, Nq, Nk, d, seed)
    scale = 1.0 / math.sqrt(d)
    out, lse = ea.attn_fwd_decode(q.to(DEV), k.to(DEV), v.to(DEV), causal=causal, window=window,
                                  scale=scale, splits=splits)
    torch.cuda.synchronize()
    assert ea.device_error() == ea.ATTN_OK
    o_ref, lse_ref = oracle.attn_ref_decode(q, k, v, causal=causal, window=window, scale=scale)
    label = f"B{B} Hq{Hq} Hkv{Hkv} Nq{Nq} Nk{Nk} d{d} c{causal} W{window} s{splits}"
    return out, lse, compare(out, lse, o_ref, lse_ref, label)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Nk", [1, 100, 128, 129, 1000, 5000])
@pytest.mark.parametrize("splits", [1, 3, 0])
def test_decode_single_query(Nk, d, splits):
    run_decode(2, 8, 2, 1, Nk, d, True, 0, splits, seed=5000 + Nk + d + splits)


@pytest.mark.parametrize("Nq,G", [(2, 4), (4, 8), (16, 8), (128, 1), (3, 1)])
@pytest.mark.parametrize("causal,window", [(True, 0), (False, 0), (True, 300), (False, 200)])
def test_decode_multi_query(Nq, G, causal, window):
    run_decode(2, 2 * G, 2, Nq, 1500, 128, causal, window, 0, seed=5100 + Nq + G + window)
    run_decode(1, G, 1, Nq, 700, 64, causal, window, 4, seed=5200 + Nq + G + window)


def test_decode_splits_agree():
    # different split counts change only the merge order: all within the same bound
    q, k, v = make_qkv_decode(4, 16, 4, 2, 3000, 128, 77)
    outs = []
    for s in (1, 2, 5, 24, 0):
        o, l = ea.attn_fwd_decode(q.to(DEV), k.to(DEV), v.to(DEV), causal=True, splits=s)
        outs.append((o.float(), l))
    torch.cuda.synchronize()
    for o, l in outs[1:]:
        assert (o - outs[0][0]).abs().max().item() <= 2e-2
        assert (l - outs[0][1]).abs().max().item() <= 1e-3


def test_decode_more_splits_than_tiles():
    run_decode(1, 4, 1, 1, 300, 64, True, 0, 50, seed=5300)   # 3 key tiles, 50 requested


def test_decode_small_workspace_rejected():
    q, k, v = make_qkv_decode(1, 4, 1, 1, 1000, 128, 3)
    need = ea.decode_workspace_size(1, 4, 1, 1, 1000, 128, 4)
    ws = torch.empty(need - 256, dtype=torch.uint8, device=DEV)
    with pytest.raises(ea.AttnError) as e:
        ea.attn_fwd_decode(q.to(DEV), k.to(DEV), v.to(DEV), splits=4, workspace=ws)
    assert e.value.code == ea.ATTN_ERR_WORKSPACE


def test_decode_workload_sampled():
    # the decode benchmark shape: B8 Hq32 Hkv8, one query per head after 8192 tokens
    from exact_self_attention_fwd_b300.inputs import DECODE_WORKLOADS
    w = DECODE_WORKLOADS["decode_8k"]
    q, k, v = make_qkv_decode(w.B, w.Hq, w.Hkv, w.Nq, w.Nk, w.d, w.seed)
    out, lse = ea.attn_fwd_decode(q.to(DEV), k.to(DEV), v.to(DEV), causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([np.arange(0, 8), np.arange(w.B * w.Hq * w.Nq - 8, w.B * w.Hq * w.Nq),
                                     np.random.default_rng(1).integers(0, w.B * w.Hq * w.Nq, 40)]))
    o_ref, l_ref = oracle.attn_ref_decode(q, k, v, causal=w.causal, scale=w.scale, rows=rows)
    compare(out.reshape(-1, w.d)[torch.from_numpy(rows).to(DEV)],
            lse.reshape(-1)[torch.from_numpy(rows).to(DEV)], o_ref, l_ref, "decode_8k")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Nk,W,splits", [(3000, 2500, 1), (2200, 0, 1), (2048, 0, 1), (4500, 0, 2), (6200, 0, 3)])
def test_decode_both_tiles_odd_and_even_tile_counts(Nk, W, splits, d):
    # up to 32 packed rows and 16 or more key tiles per split put both query tiles on each
    # split, alternating key tiles: splits of 20, 18, 16, 18 and 17 key tiles (odd and
    # even counts, tile 1 ending a step before or with tile 0)
    run_decode(2, 16, 2, 4, Nk, d, True, W, splits, seed=5600 + Nk + d + splits)
    run_decode(2, 8, 2, 1, Nk, d, True, W, splits, seed=5700 + Nk + d + splits)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("splits", [1, 2])
def test_decode_both_tiles_several_units_per_cta(d, splits):
    # 40 x 8 KV heads (x splits) units of 17 or 18 key tiles with both query tiles on each
    # split: more units than SMs, so a CTA merges one unit's two tiles (tile 0 reading
    # tile 1's O from tensor memory) and then runs the next unit, whose first P.V product
    # overwrites that O
    run_decode(40, 32, 8, 1, 2200 * splits, d, True, 0, splits, seed=5950 + d + splits)
