"""Pins for the oracle's FP8 (e4m3) block quantisation and FP8 attention (CPU only).

  codec        every one of the 256 codes decodes like torch's float8_e4m3fn; every
               bf16 value in [-448, 448] and random fp64 values encode like torch's
               round-to-nearest-even conversion
  quantiser    each block's largest magnitude comes back exactly, every element within
               half an e4m3 step (3 mantissa bits: relative 2^-4, or 2^-10 x scale for
               subnormals), scales are amax / 448
  attention    inputs that are e4m3 values already (amax 448) are reproduced exactly,
               so FP8 attention equals the plain oracle on them; with heads of very
               different magnitude, block scaling has lower error than one scale per
               tensor (the FlashAttention-3 review reports 2.6x lower RMSE for its block
               quantisation and incoherent processing on its own data)
"""
import math

import numpy as np
import pytest
import torch

import oracle


def test_decode_every_code_like_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9 and ours[0x08] == 2.0 ** -6


def test_encode_bf16_range_and_random_like_torch():
    # every bf16 value of magnitude <= 448, and random fp64 values
    bits = np.arange(1 << 16, dtype=np.uint32) << 16
    f32 = bits.view(np.float32)
    f32 = f32[np.isfinite(f32)]
    vals = f32.astype(np.float64)
    vals = vals[np.abs(vals) <= 448.0]
    rng = np.random.default_rng(3)
    vals = np.concatenate([vals, rng.uniform(-448, 448, 200000), rng.normal(0, 1e-2, 50000)])
    ours = oracle.e4m3_encode(vals)
    ref = torch.from_numpy(vals.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    # the torch conversion takes fp32: compare where the fp32 rounding does not matter
    exact32 = vals.astype(np.float32).astype(np.float64) == vals
    assert np.array_equal(ours[exact32], ref[exact32])
    # and at exact ties between codes, the even code wins
    for c in range(0x08, 0x7D):
        mid = (oracle.e4m3_decode(np.uint8(c)) + oracle.e4m3_decode(np.uint8(c + 1))) / 2
        want = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_encode(np.array([mid]))[0] == want
    assert oracle.e4m3_encode(np.array([1000.0, -1e6]))[0] == 0x7E   # saturation


def test_block_quantiser_bounds():
    g = torch.Generator().manual_seed(40)
    x = (torch.randn(3, 300, 64, generator=g) * torch.exp(torch.randn(3, 300, 1, generator=g))).bfloat16()
    codes, scales = oracle.quantize_e4m3_blocks(x, rows=128)
    assert scales.shape == (3, 3)
    deq = oracle.dequantize_e4m3_blocks(codes, scales, rows=128)
    xd = x.double().numpy()
    for h in range(3):
        for k in range(3):
            blk = xd[h, 128 * k:128 * (k + 1)]
            amax = np.abs(blk).max()
            assert math.isclose(float(scales[h, k]), float(np.float32(amax) / np.float32(448.0)), rel_tol=0)
            sc = float(scales[h, k])
            err = np.abs(deq[h, 128 * k:128 * (k + 1)] - blk)
            bound = np.maximum(np.abs(blk) * 2.0 ** -4, sc * 2.0 ** -10) * (1 + 1e-6)
            assert np.all(err <= bound)
            i = np.unravel_index(np.argmax(np.abs(blk)), blk.shape)
            assert abs(deq[h, 128 * k + i[0], i[1]] - blk[i]) <= 1e-6 * abs(blk[i])


def test_fp8_attention_exact_on_representable_inputs():
    # values that are e4m3 codes with each block's max at 448: the scale is 1 and the
    # quantisation reproduces them, so FP8 attention equals the plain oracle
    rng = np.random.default_rng(41)
    codes = rng.integers(0, 0x7E, size=(1, 2, 256, 64)).astype(np.uint8)
    codes[..., 0, 0] = 0x7E
    codes[..., 128, 0] = 0x7E
    vals = oracle.e4m3_decode(codes) * np.where(rng.random(codes.shape) < 0.5, -1, 1)
    t = torch.from_numpy(vals).float().bfloat16()
    assert np.array_equal(t.double().numpy(), vals)      # e4m3 values are bf16 values
    o8, l8, deq = oracle.attn_ref_fp8(t, t, t, causal=True, scale=2.0 ** -12)
    for dq in deq:
        assert np.array_equal(dq, vals)
    o, l = oracle.attn_ref(t, t, t, causal=True, scale=2.0 ** -12)
    assert np.array_equal(o8, o) and np.array_equal(l8, l)


def test_block_scaling_beats_tensor_scaling_with_outliers():
    # heads whose magnitudes differ by 10^4 (e4m3's normal range spans about 2^14.8):
    # one scale for the whole tensor pushes the small head into e4m3's subnormals,
    # block scales keep every block in the normal range. Measured per head, relative
    # to that head's output, the worst head's error drops.
    g = torch.Generator().manual_seed(42)
    B, H, N, d = 1, 2, 256, 64
    mag = torch.tensor([1.0, 1e-4]).view(1, H, 1, 1)
    q = (torch.randn(B, H, N, d, generator=g) * mag).bfloat16()
    k = (torch.randn(B, H, N, d, generator=g) * mag).bfloat16()
    v = (torch.randn(B, H, N, d, generator=g) * mag).bfloat16()
    o_ex, _ = oracle.attn_ref(q, k, v, causal=True, scale=0.125)
    o_blk, _, _ = oracle.attn_ref_fp8(q, k, v, causal=True, scale=0.125)
    o_ten, _, _ = oracle.attn_ref_fp8(q, k, v, causal=True, scale=0.125, per_tensor=True)

    def worst_rel_rmse(o):
        return max(float(np.sqrt(np.mean((o[0, h] - o_ex[0, h]) ** 2)) / np.sqrt(np.mean(o_ex[0, h] ** 2)))
                   for h in range(H))

    # the review's 2.6x is for FlashAttention-3's own data; here the direction is
    # asserted, with a margin (on this data the ratio is about 1.3)
    r_blk, r_ten = worst_rel_rmse(o_blk), worst_rel_rmse(o_ten)
    assert r_blk * 1.2 < r_ten, (r_blk, r_ten)


# ------------------------------------------------------------ incoherent processing
def test_hadamard_is_sylvester_and_orthogonal():
    import scipy.linalg
    for d in (1, 2, 4, 8, 16, 32, 64, 128):
        h = oracle.hadamard(d)
        assert np.array_equal(h, scipy.linalg.hadamard(d).astype(np.float64))
        assert np.array_equal(h @ h.T, d * np.eye(d))
    with pytest.raises(ValueError):
        oracle.hadamard(96)


def test_incoherent_one_hot_rows():
    # e_i M = s_i H[i, :] / sqrt(d): row i of the Hadamard matrix, with channel i's sign
    d = 128
    rng = np.random.default_rng(43)
    s = np.where(rng.random(d) < 0.5, -1.0, 1.0)
    h = oracle.hadamard(d)
    for i in (0, 1, 5, 64, 127):
        x = np.zeros((1, d))
        x[0, i] = 1.0
        y = oracle.incoherent(x, s)
        assert np.allclose(y[0], s[i] * h[i] / np.sqrt(d), atol=1e-15, rtol=0)
    # Sylvester entries (-1)^popcount(i & j)
    for i, j in ((3, 5), (127, 127), (64, 63), (96, 33)):
        assert h[i, j] == (-1) ** bin(i & j).count("1")


def test_incoherent_preserves_scores_and_attention():
    # Q' K'^T = Q M M^T K^T = Q K^T, so attention on (Q', K', V) equals attention on (Q, K, V)
    g = torch.Generator().manual_seed(44)
    B, H, N, d = 1, 2, 130, 128
    q, k, v = (torch.randn(B, H, N, d, generator=g).bfloat16() for _ in range(3))
    s = np.where(np.random.default_rng(45).random(d) < 0.5, -1.0, 1.0)
    qi, ki = oracle.incoherent(q, s), oracle.incoherent(k, s)
    assert np.allclose(qi[0, 0] @ ki[0, 0].T, q[0, 0].double().numpy() @ k[0, 0].double().numpy().T,
                       atol=1e-11, rtol=0)
    o1, l1 = oracle.attn_ref_f64in(qi, ki, v.double().numpy(), True, 0, 0.088)
    o0, l0 = oracle.attn_ref(q, k, v, causal=True, scale=0.088)
    assert np.allclose(o1, o0, atol=1e-12, rtol=0) and np.allclose(l1, l0, atol=1e-12, rtol=0)


def test_real_valued_quantiser_bounds_and_exact_case():
    g = torch.Generator().manual_seed(46)
    x = (torch.randn(2, 300, 128, generator=g) * 3).double().numpy()
    codes, scales = oracle.quantize_e4m3_blocks_f64(x, rows=128)
    deq = oracle.dequantize_e4m3_blocks(codes, scales, rows=128)
    for h in range(2):
        for kb in range(3):
            blk = x[h, 128 * kb:128 * (kb + 1)]
            sc = float(scales[h, kb])
            assert sc == np.abs(blk).max() / 448.0
            err = np.abs(deq[h, 128 * kb:128 * (kb + 1)] - blk)
            assert np.all(err <= np.maximum(np.abs(blk) * 2.0 ** -4, sc * 2.0 ** -10) * (1 + 1e-12))
    # with a block maximum of 448 both quantisers scale by exactly 1, so on bf16 inputs
    # the exact-arithmetic one and the fp32 one give the same codes
    xb = (torch.randn(1, 128, 64, generator=g) * 40).bfloat16()
    xb[0, 0, 0] = 448.0
    xb = xb.clamp(-448, 448)
    c32, s32 = oracle.quantize_e4m3_blocks(xb, rows=128)
    c64, s64 = oracle.quantize_e4m3_blocks_f64(xb.double().numpy(), rows=128)
    assert np.array_equal(c32, c64) and float(s32[0, 0]) == float(s64[0, 0]) == 1.0


def test_incoherent_processing_helps_with_outlier_channels():
    # a few channels of Q and K far larger than the rest: with block scales the small
    # channels lose their precision to the outliers' scale; the rotation spreads each
    # outlier over all channels first. The error of FP8 attention against exact
    # attention drops (the direction the review states; the margin is this data's).
    g = torch.Generator().manual_seed(47)
    B, H, N, d = 1, 2, 256, 128
    boost = torch.ones(d)
    boost[[7, 70]] = 60.0
    q = (torch.randn(B, H, N, d, generator=g) * boost).bfloat16()
    k = (torch.randn(B, H, N, d, generator=g) * boost * 0.02).bfloat16()
    v = torch.randn(B, H, N, d, generator=g).bfloat16()
    s = np.where(np.random.default_rng(48).random(d) < 0.5, -1.0, 1.0)
    o_ex, _ = oracle.attn_ref(q, k, v, causal=True, scale=0.088)
    o_blk, _, _ = oracle.attn_ref_fp8(q, k, v, causal=True, scale=0.088)
    o_inc, _, _ = oracle.attn_ref_fp8(q, k, v, causal=True, scale=0.088, signs=s)
    e_blk = float(np.sqrt(np.mean((o_blk - o_ex) ** 2)))
    e_inc = float(np.sqrt(np.mean((o_inc - o_ex) ** 2)))
    assert e_inc * 1.5 < e_blk, (e_inc, e_blk)
