"""The FP8 (e4m3) path through the C ABI: block quantisation must match the oracle's
bit for bit (integer codes and fp32 scales), and attention on the e4m3 operands is
compared with the fp64 oracle on the dequantised values.

Tolerance of the FP8 attention (from the arithmetic): S is exact up to fp32
accumulation, so the LSE keeps the 1e-3 relative bar. P is rounded to e4m3 (3 mantissa
bits: relative error delta <= 2^-4) for the P.V product and O is normalised by the
rounded weights, so O - O_ref = sum_j w_j (delta_j - mean delta) (v_j - O_ref) / (1 +
mean delta); per element that is at most 2 * 2^-4 * 2 max|v| / (1 - 2^-4), and its root
mean square is bounded by 2^-4 * RMS(v).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import exact_self_attention_fwd_b300 as ea
from exact_self_attention_fwd_b300.inputs import make_qkv

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
MAX_FRAC = 2 * 2.0 ** -4 * 2 / (1 - 2.0 ** -4)


@pytest.mark.parametrize("shape", [(1, 2, 128, 128), (2, 3, 300, 128), (1, 4, 1000, 64), (2, 1, 77, 64)])
def test_quantize_matches_oracle_bit_for_bit(shape):
    g = torch.Generator().manual_seed(sum(shape))
    x = (torch.randn(shape, generator=g) * torch.exp(2 * torch.randn(shape[:-1] + (1,), generator=g))).bfloat16()
    x[..., 0, 0] = 0.0
    codes, scales = ea.quantize_e4m3(x.to(DEV))
    torch.cuda.synchronize()
    c_ref, s_ref = oracle.quantize_e4m3_blocks(x, rows=128)
    assert np.array_equal(codes.cpu().numpy(), c_ref)
    assert np.array_equal(scales.cpu().numpy().reshape(s_ref.shape), s_ref)


def test_quantize_zero_block():
    x = torch.zeros(1, 256, 128, dtype=torch.bfloat16, device=DEV)
    x[0, 200, 3] = 2.0
    codes, scales = ea.quantize_e4m3(x)
    torch.cuda.synchronize()
    assert scales[0, 0].item() == 1.0 and codes[0, :128].eq(0).all()
    assert scales[0, 1].item() == np.float32(2.0) / np.float32(448.0)


def run_fp8(B, Hq, Hkv, N, causal, window, seed):
    d = 128
    q, k, v = make_qkv(B, Hq, Hkv, N, d, seed)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    (q8, qs), (k8, ks), (v8, vs) = ea.quantize_e4m3(qd), ea.quantize_e4m3(kd), ea.quantize_e4m3(vd)
    scale = 1.0 / math.sqrt(d)
    out, lse = ea.attn_fwd_fp8(q8, k8, v8, qs, ks, vs, causal=causal, window=window, scale=scale)
    torch.cuda.synchronize()
    assert ea.device_error() == ea.ATTN_OK
    # the oracle quantises the same inputs with its own codec (bit-identical to the GPU's,
    # which test_quantize_matches_oracle_bit_for_bit checks) and attends in fp64
    o_ref, l_ref, deq = oracle.attn_ref_fp8(q, k, v, causal=causal, window=window, scale=scale)
    o = out.float().cpu().double().numpy()
    l = lse.cpu().double().numpy()
    assert np.isfinite(o).all() and np.isfinite(l).all()
    lerr = np.abs(l - l_ref) / np.maximum(1.0, np.abs(l_ref))
    assert lerr.max() <= 1e-3, f"LSE rel err {lerr.max():.3g}"
    vmax = np.abs(deq[2]).max()
    err = np.abs(o - o_ref)
    assert err.max() <= MAX_FRAC * vmax + 2.0 ** -6, f"max |dO| {err.max():.3g}"
    rmse = float(np.sqrt(np.mean(err ** 2)))
    assert rmse <= 2.0 ** -4 * float(np.sqrt(np.mean(deq[2] ** 2))), f"RMSE {rmse:.3g}"
    return err.max(), rmse


@pytest.mark.parametrize("N", [128, 129, 300, 1000])
@pytest.mark.parametrize("causal,window", [(False, 0), (True, 0), (True, 200), (False, 150)])
def test_fp8_attention_vs_oracle(N, causal, window):
    mx, rmse = run_fp8(2, 4, 2, N, causal, window, seed=6000 + N + window)
    print(N, causal, window, mx, rmse)


def test_fp8_many_units():
    run_fp8(2, 32, 8, 2048, True, 0, seed=6100)


# ------------------------------------------------------------ incoherent processing
# The rotated values y = (x o s) H are formed in fp32 by 7 butterfly stages; each output
# is a sum of 128 signed bf16 inputs, so |y_fp32 - y| <= gamma_7 sum_i |x_i| with
# gamma_7 = 7u / (1 - 7u), u = 2^-24, and the block's amax moves by at most the block's
# largest such bound. A code may therefore differ from the oracle's exact one only where
# the exact target t = y 448 / amax lies within that error of the rounding boundary
# between the two codes (there both codes are correct roundings); everywhere else it
# must be identical.
U = 2.0 ** -24
GAMMA7 = 7 * U / (1 - 7 * U)


def check_hadamard_codes(x, signs, codes, scales):
    xv = x.double().numpy()
    *lead, N, d = xv.shape
    BH = int(np.prod(lead))
    xv = xv.reshape(BH, N, d)
    yn = oracle.incoherent(xv, signs)                     # x M, fp64
    c_ref, s_ref = oracle.quantize_e4m3_blocks_f64(yn, rows=128)
    cg = codes.cpu().numpy().reshape(BH, N, d)
    sg = scales.cpu().numpy().reshape(s_ref.shape).astype(np.float64)
    yu = yn * np.sqrt(d)                                  # the unnormalised sums the kernel forms
    e_row = GAMMA7 * np.abs(xv).sum(-1, keepdims=True)    # [BH, N, 1]
    nblk = s_ref.shape[1]
    flips = 0
    for h in range(BH):
        for kb in range(nblk):
            r0, r1 = 128 * kb, min(N, 128 * (kb + 1))
            y = yu[h, r0:r1]
            amax = np.abs(y).max()
            if amax == 0:
                assert sg[h, kb] == 1.0 and not cg[h, r0:r1].any()
                continue
            e_blk = e_row[h, r0:r1].max()
            assert abs(sg[h, kb] - s_ref[h, kb]) <= s_ref[h, kb] * (1.01 * e_blk / amax + 4 * U), (h, kb)
            t = y * (448.0 / amax)
            eta = 1.01 * (448.0 / amax) * (e_row[h, r0:r1] + np.abs(y) * e_blk / amax) + 4 * U * np.abs(t)
            a, b = c_ref[h, r0:r1], cg[h, r0:r1]
            diff = a != b
            if not diff.any():
                continue
            va, vb = oracle.e4m3_decode(a[diff]), oracle.e4m3_decode(b[diff])
            same_value = va == vb                          # +0 and -0
            adjacent = ((a[diff] & 0x80) == (b[diff] & 0x80)) & (
                np.abs((a[diff] & 0x7F).astype(int) - (b[diff] & 0x7F).astype(int)) == 1)
            near = np.abs(t[diff] - (va + vb) / 2) <= eta[diff]
            ok = same_value | (adjacent & near)
            assert ok.all(), f"head {h} block {kb}: {int((~ok).sum())} codes off beyond the fp32 bound"
            flips += int((~same_value).sum())
    return flips


@pytest.mark.parametrize("shape", [(1, 2, 128, 128), (2, 3, 300, 128), (1, 1, 77, 128)])
def test_hadamard_quantize_vs_oracle(shape):
    from exact_self_attention_fwd_b300.inputs import make_signs
    g = torch.Generator().manual_seed(sum(shape) + 1)
    x = (torch.randn(shape, generator=g) * torch.exp(2 * torch.randn(shape[:-1] + (1,), generator=g))).bfloat16()
    x[..., 5, :] = 0.0                                     # an all-zero row
    signs = make_signs(128, sum(shape))
    codes, scales = ea.quantize_e4m3_hadamard(x.to(DEV), signs)
    torch.cuda.synchronize()
    flips = check_hadamard_codes(x, signs, codes, scales)
    assert flips <= 1e-4 * x.numel(), flips


def test_hadamard_quantize_zero_block_and_outliers():
    from exact_self_attention_fwd_b300.inputs import make_signs
    x = torch.zeros(1, 256, 128, dtype=torch.bfloat16)
    g = torch.Generator().manual_seed(3)
    x[0, 128:] = torch.randn(128, 128, generator=g).bfloat16()
    x[0, 130, 17] = 300.0                                  # one outlier channel element
    signs = make_signs(128, 9)
    codes, scales = ea.quantize_e4m3_hadamard(x.to(DEV), signs)
    torch.cuda.synchronize()
    assert scales[0, 0].item() == 1.0 and codes[0, :128].eq(0).all()
    check_hadamard_codes(x, signs, codes, scales)


def run_fp8_hadamard(B, Hq, Hkv, N, causal, window, seed):
    from exact_self_attention_fwd_b300.inputs import make_signs
    d = 128
    q, k, v = make_qkv(B, Hq, Hkv, N, d, seed)
    signs = make_signs(d, seed + 1)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    (q8, qs), (k8, ks) = ea.quantize_e4m3_hadamard(qd, signs), ea.quantize_e4m3_hadamard(kd, signs)
    v8, vs = ea.quantize_e4m3(vd)
    scale = 1.0 / math.sqrt(d)
    out, lse = ea.attn_fwd_fp8(q8, k8, v8, qs, ks, vs, causal=causal, window=window, scale=scale)
    torch.cuda.synchronize()
    assert ea.device_error() == ea.ATTN_OK
    o_ref, l_ref, deq = oracle.attn_ref_fp8(q, k, v, causal=causal, window=window, scale=scale, signs=signs)
    o = out.float().cpu().double().numpy()
    l = lse.cpu().double().numpy()
    assert np.isfinite(o).all() and np.isfinite(l).all()
    lerr = np.abs(l - l_ref) / np.maximum(1.0, np.abs(l_ref))
    assert lerr.max() <= 1e-3, f"LSE rel err {lerr.max():.3g}"
    vmax = np.abs(deq[2]).max()
    err = np.abs(o - o_ref)
    assert err.max() <= MAX_FRAC * vmax + 2.0 ** -6, f"max |dO| {err.max():.3g}"
    rmse = float(np.sqrt(np.mean(err ** 2)))
    assert rmse <= 2.0 ** -4 * float(np.sqrt(np.mean(deq[2] ** 2))), f"RMSE {rmse:.3g}"
    return err.max(), rmse


@pytest.mark.parametrize("N,causal,window", [(128, False, 0), (300, True, 0), (1000, True, 200), (257, False, 90)])
def test_fp8_hadamard_attention_vs_oracle(N, causal, window):
    run_fp8_hadamard(2, 4, 2, N, causal, window, seed=6200 + N)
