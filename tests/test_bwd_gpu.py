"""The backward pass (attn_bwd, through the C ABI) against the fp64 oracle's gradients.

The backward takes the forward's O and LSE as inputs. The parity tests give it the
oracle's O rounded to bf16 and the oracle's LSE rounded to fp32 (what a bf16/fp32
forward returns at best), and compare with the oracle's gradients for that same O
(oracle.attn_ref_bwd(o=...): the row term dO_i . O_i from the given O). Tolerance,
derived from the arithmetic of the CUDA path; u = 2^-8 is the unit roundoff of bf16
(8 significant bits, round to nearest even):
  * dV = P^T dO: P is rounded to bf16 for the product (relative error <= u per term)
    and the result once more (<= u). So, elementwise and rigorously,
        |dV - ref| <= 3u A + 1e-6,   A = sum_i P_ij |dO_i|
    (A is the oracle's dV for |dO|: P >= 0 makes it the sum of the terms' magnitudes;
    the third u covers fp32 accumulation, exp2 and the fp32 LSE).
  * dQ, dK: dS is rounded to bf16 (u per term) and the result once more (u); D and dP
    are fp32 sums of exact bf16 products. Per row r:
        ||g_r - ref_r|| <= 5u ||ref_r|| + 2e-3 rms + 1e-6
    (5u leaves room for sums whose terms partly cancel; rms is the largest
    root-mean-square row norm of the three exact gradients, so the second term covers
    rows whose exact gradient is zero, like dQ of a query that sees one key, where
    fp32 rounding of dP - D leaves a residual). Tensor: ||g - ref||_F <= 1e-2 ||ref||_F.
A wrong mask, index, scale or head map moves whole rows by O(1) relative.

The pipeline tests run the GPU forward and feed its O to the backward. Its O carries up
to 2u of sum_j P_ij |V_j| per element (P rounded in the P.V product, O on output), so
|D_i - D_exact| <= delta_i = 2u sum_c |dO_ic| Obar_ic (Obar: the oracle's forward for
|V|), which enters dS_ij as P_ij delta_i and adds, per row, at most
scale delta_i max_j ||K_j|| to dQ_i and scale colsum_j max_i (delta_i ||Q_i||) to dK_j
(colsum_j = sum_i P_ij, the oracle's dV for dO = 1), compared with the exact gradients.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
import exact_self_attention_fwd_b300 as ea
from exact_self_attention_fwd_b300.inputs import make_dout, make_qkv

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
U = 2.0 ** -8
ROW_REL = 5 * U
ROW_FLOOR = 2e-3
FRO_REL = 1e-2


def _np(t):
    return t.detach().float().cpu().double().numpy()


def rms_rows(ref):
    r2 = (ref ** 2).reshape(-1, ref.shape[-1]).sum(1)
    return float(np.sqrt(r2.mean())) if r2.size else 0.0


def check_rows(g, ref, name, label, rms, extra):
    assert np.isfinite(g).all(), f"{label}: non-finite {name}"
    d = g.shape[-1]
    e = np.sqrt(((g - ref) ** 2).reshape(-1, d).sum(1))
    r = np.sqrt((ref ** 2).reshape(-1, d).sum(1))
    extra = np.asarray(extra, dtype=np.float64).reshape(-1)
    bound = ROW_REL * r + extra + ROW_FLOOR * rms + 1e-6
    bad = np.nonzero(e > bound)[0]
    assert bad.size == 0, (f"{label}: {bad.size} rows of {name} off, first {bad[:5]}: "
                           f"err {e[bad[:5]]} ref {r[bad[:5]]}")
    fro = float(np.sqrt((e ** 2).sum())), float(np.sqrt((r ** 2).sum()))
    assert fro[0] <= FRO_REL * fro[1] + float(np.sqrt((extra ** 2).sum())) + ROW_FLOOR * rms * np.sqrt(r.size) + 1e-6, f"{label}: {name} rel Frobenius {fro[0] / max(fro[1], 1e-30):.3g}"
    return fro[0] / max(fro[1], 1e-30)


def d_term(q, k, v, do, causal, window, scale, key_len):
    """Row bounds on the error that D = rowsum(dO o O_bf16) carries into dQ and dK."""
    B, Hq, N, d = q.shape
    Hkv = k.shape[1]
    G = Hq // Hkv
    obar, _ = oracle.attn_ref(q, k, v.abs(), causal=causal, window=window, scale=scale, key_len=key_len)
    delta = 2 * U * (do.double().abs().numpy() * obar).sum(-1)                    # [B,Hq,N]
    knorm = np.sqrt((k.double().numpy() ** 2).sum(-1)).max(-1)                  # [B,Hkv]
    eq = scale * delta * np.repeat(knorm, G, axis=1)[..., None]
    qn = np.sqrt((q.double().numpy() ** 2).sum(-1))                             # [B,Hq,N]
    w = (delta * qn).reshape(B, Hkv, G * N).max(-1)                             # [B,Hkv]
    _, _, colsum = oracle.attn_ref_bwd(q, k, v, torch.ones_like(do), causal=causal, window=window,
                                       scale=scale, key_len=key_len)
    ek = scale * colsum[..., 0] * w[..., None]
    return eq, ek


def check_bwd(B, Hq, Hkv, N, d, causal, window, seed, key_len=None, q_head0_scale=1.0, scale=None,
              pipeline=False):
    q, k, v = make_qkv(B, Hq, Hkv, N, d, seed, q_head0_scale)
    do = make_dout(B, Hq, N, d, seed + 7)
    scale = scale or 1.0 / math.sqrt(d)
    kl = None if key_len is None else torch.tensor(key_len, dtype=torch.int32, device=DEV)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    if pipeline:
        out, lse = ea.attn_fwd(qd, kd, vd, causal=causal, window=window, scale=scale, key_len=kl)
        o_given = None
    else:
        o_ref, lse_ref = oracle.attn_ref(q, k, v, causal=causal, window=window, scale=scale, key_len=key_len)
        out = torch.from_numpy(o_ref).to(torch.bfloat16).to(DEV)
        lse = torch.from_numpy(lse_ref).float().to(DEV)
        o_given = out.double().cpu()
    ws = torch.full((ea.bwd_workspace_size(B, Hq, N, d),), 0xFF, dtype=torch.uint8, device=DEV)  # NaN fill
    dq, dk, dv = ea.attn_bwd(qd, kd, vd, out, lse, dod, causal=causal, window=window, scale=scale,
                             key_len=kl, workspace=ws)
    torch.cuda.synchronize()
    assert ea.device_error() == ea.ATTN_OK
    rq, rk, rv = oracle.attn_ref_bwd(q, k, v, do, causal=causal, window=window, scale=scale,
                                     key_len=key_len, o=o_given)
    label = f"B{B} Hq{Hq} Hkv{Hkv} N{N} d{d} c{causal} W{window} L{key_len}"
    if not pipeline:
        # D = rowsum(dO o O) from the given bf16 values: exact products, an fp32 sum of d
        # of them (error <= d 2^-24 of the sum of magnitudes)
        prod = do.double().numpy() * o_given.numpy()
        dsum = _np(ea.bwd_row_sums(ws, B, Hq, N))
        assert np.all(np.abs(dsum - prod.sum(-1)) <= d * 2.0 ** -24 * np.abs(prod).sum(-1) + 1e-30), \
            f"{label}: D differs from rowsum(dO o O)"
    rms = max(rms_rows(rq), rms_rows(rk), rms_rows(rv))
    if pipeline:
        eq, ek = d_term(q, k, v, do, causal, window, scale, key_len)
    else:
        eq, ek = np.zeros(rq.shape[:-1]), np.zeros(rk.shape[:-1])
    res = {n: check_rows(_np(g), r, n, label, rms, x)
           for n, g, r, x in (("dq", dq, rq, eq), ("dk", dk, rk, ek), ("dv", dv, rv, np.zeros(rv.shape[:-1])))}
    # rigorous elementwise bound on dV from the magnitudes of its terms
    _, _, av = oracle.attn_ref_bwd(q, k, v, do.abs(), causal=causal, window=window, scale=scale,
                                   key_len=key_len)
    err = np.abs(_np(dv) - rv)
    worst = float((err - (3 * U * av + 1e-6)).max()) if err.size else -1.0
    assert worst <= 0.0, f"{label}: dV exceeds 3u x sum of |terms| by {worst:.3g}"
    return res


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 2, 127, 128, 129, 197, 300])
def test_bwd_lengths(N, d, causal):
    check_bwd(1, 2, 2, N, d, causal, 0, seed=5000 + N + d + int(causal))


@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("causal", [False, True])
def test_bwd_gqa(G, causal):
    check_bwd(2, 8, 8 // G, 260, 128, causal, 0, seed=5100 + G)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("W", [1, 100, 128, 129, 300, 1000])
def test_bwd_causal_window(W, d):
    check_bwd(1, 4, 2, 600, d, True, W, seed=5200 + W)


@pytest.mark.parametrize("W", [1, 64, 130, 400])
def test_bwd_symmetric_window(W):
    check_bwd(1, 2, 1, 520, 64, False, W, seed=5300 + W)


@pytest.mark.parametrize("causal,W", [(False, 0), (True, 0), (True, 90), (False, 90)])
def test_bwd_padding(causal, W):
    check_bwd(3, 4, 2, 300, 128, causal, W, seed=5400 + W, key_len=[300, 131, 0])


def test_bwd_softmax_range():
    # the GPT-2-small-shaped recipe's head-0 query x4 makes peaky rows
    check_bwd(1, 3, 3, 512, 64, True, 0, seed=5500, q_head0_scale=4.0)


def test_bwd_multi_tile():
    check_bwd(1, 4, 1, 1100, 128, True, 0, seed=5600)
    check_bwd(1, 2, 2, 1000, 64, False, 0, seed=5601)


@pytest.mark.parametrize("d,Hkv", [(64, 8), (128, 2)])
def test_bwd_many_units_per_cta_with_padding(d, Hkv):
    """More units than SMs (320 dQ units; 320 dK/dV units at d = 64), so each CTA runs
    several and alternates between its accumulator sets, with padded batches whose tiles
    past their length have nothing to stream (those units write zeros between units that
    accumulate)."""
    check_bwd(8, 8, Hkv, 640, d, True, 0, seed=5900 + d, key_len=[640, 200, 0, 513, 128, 1, 640, 300])


# ------------------------------------------------------------ GPU forward feeding the backward
@pytest.mark.parametrize("case", [
    (1, 2, 2, 197, 64, False, 0, None),
    (2, 8, 2, 300, 128, True, 0, None),
    (1, 4, 2, 600, 128, True, 128, None),
    (1, 2, 1, 520, 64, False, 130, None),
    (3, 4, 2, 300, 128, True, 90, [300, 131, 0]),
])
def test_bwd_pipeline(case):
    B, Hq, Hkv, N, d, causal, W, kl = case
    check_bwd(B, Hq, Hkv, N, d, causal, W, seed=5800 + N, key_len=kl, pipeline=True)


def test_bwd_rejects_bad_arguments():
    q, k, v = (t.to(DEV) for t in make_qkv(1, 2, 1, 64, 64, 1))
    out, lse = ea.attn_fwd(q, k, v)
    with pytest.raises(ValueError):
        ea.attn_bwd(q, k, v, out, lse, out[:, :1].contiguous())
    L = ea.load()
    need = ea.bwd_workspace_size(1, 2, 64, 64)
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    args = [q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), out.data_ptr(),
            q.data_ptr(), k.data_ptr(), v.data_ptr(), None, 1, 2, 1, 64, 64, 0, 0, 0.125, ws.data_ptr(), need, None]
    bad = list(args)
    bad[6] = None
    assert L.attn_bwd(*bad) == ea.ATTN_ERR_NULLPTR
    bad = list(args)
    bad[14] = 96
    assert L.attn_bwd(*bad) == ea.ATTN_ERR_UNSUPPORTED
    bad = list(args)
    bad[19] = need - 1
    assert L.attn_bwd(*bad) == ea.ATTN_ERR_WORKSPACE
    assert L.attn_bwd(*args) == ea.ATTN_OK
    torch.cuda.synchronize()


# ------------------------------------------------------------ full-size workloads
@pytest.mark.parametrize("name", ["gpt2_small", "gqa_8k", "swa_16k"])
def test_bwd_full_size_sampled_dq_rows(name):
    """The benchmark's backward configuration (GPU forward feeding attn_bwd) at the
    workload's full size. dq rows are checked one by one against the oracle's row
    gradients with the pipeline bound (see the module docstring): 5u ||ref|| + the D-term
    scale delta_i max_j ||K_j|| + 2e-3 rms. dk and dv are not computable row by row
    (each needs every query's weights); the smaller parity cases above cover them."""
    from exact_self_attention_fwd_b300.inputs import WORKLOADS, make_workload
    from parity import sample_rows
    w = WORKLOADS[name]
    q, k, v = make_workload(w)
    do = make_dout(w.B, w.Hq, w.N, w.d, w.seed + 100)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    out, lse = ea.attn_fwd(qd, kd, vd, causal=w.causal, window=w.window, scale=w.scale)
    dq, dk, dv = ea.attn_bwd(qd, kd, vd, out, lse, dod, causal=w.causal, window=w.window, scale=w.scale)
    torch.cuda.synchronize()
    assert ea.device_error() == ea.ATTN_OK
    for t in (dq, dk, dv):
        assert torch.isfinite(t).all()
    rows = sample_rows(w.B, w.Hq, w.N, w.window, 120, seed=11)
    ref = oracle.attn_ref_bwd_dq_rows(q, k, v, do, rows, causal=w.causal, window=w.window, scale=w.scale)
    got = dq.reshape(-1, w.d)[torch.from_numpy(rows).to(DEV)].float().cpu().double().numpy()
    # D-term: delta_i = 2u sum_c |dO_ic| Obar_ic, Obar the oracle's forward for |V|
    obar, _ = oracle.attn_ref_rows(q, k, v.abs(), w.causal, w.window, w.scale, rows)
    dabs = do.reshape(-1, w.d)[torch.from_numpy(rows)].double().abs().numpy()
    delta = 2 * U * (dabs * obar.reshape(len(rows), w.d)).sum(-1)
    knorm = np.sqrt((k.double().numpy() ** 2).sum(-1)).max()
    e = np.sqrt(((got - ref) ** 2).sum(-1))
    r = np.sqrt((ref ** 2).sum(-1))
    rms = float(np.sqrt((r ** 2).mean()))
    bound = ROW_REL * r + w.scale * delta * knorm + ROW_FLOOR * rms + 1e-6
    bad = np.nonzero(e > bound)[0]
    assert bad.size == 0, f"{name}: {bad.size} dq rows off, first {rows[bad[:5]]}: err {e[bad[:5]]} ref {r[bad[:5]]}"


@pytest.mark.parametrize("name,b,kv", [("gqa_8k", 1, 5), ("swa_16k", 0, 11)])
def test_bwd_full_size_one_group_every_element(name, b, kv):
    """The workload at full size, and every element of dK and dV (and dQ) of one
    (batch, KV head) group against the oracle's gradients for that group. The group's
    query heads get the oracle's O rounded to bf16 and its LSE rounded to fp32 (the
    other heads keep the GPU forward's, which the group's gradients do not read), and
    the tolerance is the module's: rows within 5u ||ref|| + 2e-3 rms, dV elementwise
    within 3u of the sum of its terms' magnitudes."""
    from exact_self_attention_fwd_b300.inputs import WORKLOADS, make_workload
    w = WORKLOADS[name]
    q, k, v = make_workload(w)
    do = make_dout(w.B, w.Hq, w.N, w.d, w.seed + 100)
    G = w.group
    hs = slice(kv * G, (kv + 1) * G)
    qg, dog = q[b:b + 1, hs].contiguous(), do[b:b + 1, hs].contiguous()
    kg, vg = k[b:b + 1, kv:kv + 1].contiguous(), v[b:b + 1, kv:kv + 1].contiguous()
    o_g, lse_g = oracle.attn_ref(qg, kg, vg, causal=w.causal, window=w.window, scale=w.scale)
    o_g16 = torch.from_numpy(o_g).to(torch.bfloat16)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    out, lse = ea.attn_fwd(qd, kd, vd, causal=w.causal, window=w.window, scale=w.scale)
    out[b, hs] = o_g16[0].to(DEV)
    lse[b, hs] = torch.from_numpy(lse_g[0]).float().to(DEV)
    dq, dk, dv = ea.attn_bwd(qd, kd, vd, out, lse, dod, causal=w.causal, window=w.window, scale=w.scale)
    torch.cuda.synchronize()
    assert ea.device_error() == ea.ATTN_OK
    rq, rk, rv = oracle.attn_ref_bwd(qg, kg, vg, dog, causal=w.causal, window=w.window, scale=w.scale,
                                     o=o_g16.double())
    rms = max(rms_rows(rq), rms_rows(rk), rms_rows(rv))
    label = f"{name} group b{b} kv{kv}"
    gq, gk, gv = _np(dq[b:b + 1, hs]), _np(dk[b:b + 1, kv:kv + 1]), _np(dv[b:b + 1, kv:kv + 1])
    res = {n: check_rows(g, r, n, label, rms, np.zeros(r.shape[:-1]))
           for n, g, r in (("dq", gq, rq), ("dk", gk, rk), ("dv", gv, rv))}
    _, _, av = oracle.attn_ref_bwd(qg, kg, vg, dog.abs(), causal=w.causal, window=w.window, scale=w.scale)
    worst = float((np.abs(gv - rv) - (3 * U * av + 1e-6)).max())
    assert worst <= 0.0, f"{label}: dV exceeds 3u x sum of |terms| by {worst:.3g}"
    print(label, res)


def test_bwd_is_deterministic_and_stream_ordered():
    # no atomics: two runs give identical bits, also on a side stream
    q, k, v = make_qkv(2, 8, 2, 700, 128, 5900)
    do = make_dout(2, 8, 700, 128, 5901)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    out, lse = ea.attn_fwd(qd, kd, vd, causal=True)
    a = ea.attn_bwd(qd, kd, vd, out, lse, dod, causal=True)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        b = ea.attn_bwd(qd, kd, vd, out, lse, dod, causal=True, stream=side)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x, y)
