"""Pins for the oracle's backward pass (CPU only): torch autograd through fp64
scaled_dot_product_attention with the same boolean mask (an independent library
routine), central finite differences of the oracle's own forward (the gradient's
definition), and invariants of the softmax gradient."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle


def _mask(N, causal, W, L=None):
    i = torch.arange(N).view(N, 1)
    j = torch.arange(N).view(1, N)
    m = torch.ones(N, N, dtype=torch.bool)
    if L is not None:
        m &= (i < L) & (j < L)
    if causal:
        m &= j <= i
    if W:
        m &= (i - j) < W
        if not causal:
            m &= (j - i) < W
    return m


@pytest.mark.parametrize("causal,W", [(False, 0), (True, 0), (True, 5), (False, 4)])
def test_bwd_matches_torch_autograd(causal, W):
    g = torch.Generator().manual_seed(50 + W)
    B, Hq, Hkv, N, d = 2, 4, 2, 37, 16
    q = torch.randn(B, Hq, N, d, generator=g).bfloat16()
    k = torch.randn(B, Hkv, N, d, generator=g).bfloat16()
    v = torch.randn(B, Hkv, N, d, generator=g).bfloat16()
    do = torch.randn(B, Hq, N, d, generator=g).bfloat16()
    scale = 0.3
    dq, dk, dv = oracle.attn_ref_bwd(q, k, v, do, causal=causal, window=W, scale=scale)
    G = Hq // Hkv
    qt = q.double().requires_grad_()
    kt = k.double().requires_grad_()
    vt = v.double().requires_grad_()
    o = F.scaled_dot_product_attention(qt, kt.repeat_interleave(G, 1), vt.repeat_interleave(G, 1),
                                       attn_mask=_mask(N, causal, W), scale=scale)
    o.backward(do.double())
    np.testing.assert_allclose(dq, qt.grad.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dk, kt.grad.numpy(), rtol=0, atol=1e-11)
    np.testing.assert_allclose(dv, vt.grad.numpy(), rtol=0, atol=1e-11)


def test_bwd_padding_matches_torch_on_valid_part():
    g = torch.Generator().manual_seed(55)
    B, H, N, d = 2, 2, 30, 8
    q, k, v, do = (torch.randn(B, H, N, d, generator=g).bfloat16() for _ in range(4))
    key_len = [30, 17]
    dq, dk, dv = oracle.attn_ref_bwd(q, k, v, do, causal=True, scale=0.5, key_len=key_len)
    for b, L in enumerate(key_len):
        qt = q[b:b + 1, :, :L].double().requires_grad_()
        kt = k[b:b + 1, :, :L].double().requires_grad_()
        vt = v[b:b + 1, :, :L].double().requires_grad_()
        o = F.scaled_dot_product_attention(qt, kt, vt, is_causal=True, scale=0.5)
        o.backward(do[b:b + 1, :, :L].double())
        np.testing.assert_allclose(dq[b, :, :L], qt.grad[0].numpy(), atol=1e-11, rtol=0)
        np.testing.assert_allclose(dk[b, :, :L], kt.grad[0].numpy(), atol=1e-11, rtol=0)
        np.testing.assert_allclose(dv[b, :, :L], vt.grad[0].numpy(), atol=1e-11, rtol=0)
        assert not dq[b, :, L:].any() and not dk[b, :, L:].any() and not dv[b, :, L:].any()


def test_bwd_finite_differences():
    # L = sum(do * o): dL/dx from central differences of the oracle's forward, in fp64
    # on inputs that are bf16 values (the step is far below their spacing, so the
    # perturbed inputs are not rounded: the oracle's fp64-input forward is used)
    g = torch.Generator().manual_seed(56)
    B, Hq, Hkv, N, d = 1, 2, 1, 9, 4
    q = torch.randn(B, Hq, N, d, generator=g).bfloat16()
    k = torch.randn(B, Hkv, N, d, generator=g).bfloat16()
    v = torch.randn(B, Hkv, N, d, generator=g).bfloat16()
    do = torch.randn(B, Hq, N, d, generator=g).bfloat16()
    scale, causal, W = 0.7, True, 4
    dq, dk, dv = oracle.attn_ref_bwd(q, k, v, do, causal=causal, window=W, scale=scale)
    base = [t.double().numpy() for t in (q, k, v)]
    dod = do.double().numpy()
    G = Hq // Hkv

    def loss(qq, kk, vv):
        o, _ = oracle.attn_ref_f64in(qq, kk, vv, causal, W, scale)
        return float(np.sum(o * dod))

    h = 1e-6
    for which, grad in ((0, dq), (1, dk), (2, dv)):
        x = base[which]
        for idx in [(0, 0, 0, 0), (0, 0, 3, 2), (0, x.shape[1] - 1, N - 1, d - 1), (0, 0, N // 2, 1)]:
            plus = [b.copy() for b in base]
            minus = [b.copy() for b in base]
            plus[which][idx] += h
            minus[which][idx] -= h
            fd = (loss(*plus) - loss(*minus)) / (2 * h)
            assert abs(fd - grad[idx]) <= 1e-6 * max(1.0, abs(fd)), (which, idx, fd, grad[idx])


def test_bwd_invariants():
    # constant upstream gradient c on every row: dp_ij = c . v_j and the softmax
    # gradient removes any part of dp that is constant across j; with do = 0, every
    # gradient is zero; dv sums each query row's weights, so sum_j dv_j = sum_i do_i
    g = torch.Generator().manual_seed(57)
    B, H, N, d = 1, 2, 20, 8
    q, k, v = (torch.randn(B, H, N, d, generator=g).bfloat16() for _ in range(3))
    zero = torch.zeros(B, H, N, d, dtype=torch.bfloat16)
    dq, dk, dv = oracle.attn_ref_bwd(q, k, v, zero, causal=True, scale=0.25)
    assert not dq.any() and not dk.any() and not dv.any()
    do = torch.randn(B, H, N, d, generator=g).bfloat16()
    _, _, dv = oracle.attn_ref_bwd(q, k, v, do, causal=True, scale=0.25)
    np.testing.assert_allclose(dv.sum(axis=2), do.double().numpy().sum(axis=2), atol=1e-12, rtol=0)
    # v constant across keys: o does not depend on q or k, so dq = dk = 0
    vc = torch.randn(B, H, 1, d, generator=g).bfloat16().expand(B, H, N, d).contiguous()
    dq, dk, _ = oracle.attn_ref_bwd(q, k, vc, do, causal=False, scale=0.25)
    assert np.abs(dq).max() < 1e-12 and np.abs(dk).max() < 1e-12


def test_bwd_given_exact_o_equals_chain_rule():
    # do_i . o_i equals sum_j p_ij dp_ij when o is the exact output
    g = torch.Generator().manual_seed(58)
    B, Hq, Hkv, N, d = 2, 4, 2, 37, 16
    q = torch.randn(B, Hq, N, d, generator=g).bfloat16()
    k, v = (torch.randn(B, Hkv, N, d, generator=g).bfloat16() for _ in range(2))
    do = torch.randn(B, Hq, N, d, generator=g).bfloat16()
    for causal, W, kl in ((True, 0, None), (False, 5, [37, 11]), (True, 9, [20, 37])):
        o, _ = oracle.attn_ref(q, k, v, causal=causal, window=W, scale=0.3, key_len=kl)
        a = oracle.attn_ref_bwd(q, k, v, do, causal=causal, window=W, scale=0.3, key_len=kl)
        b = oracle.attn_ref_bwd(q, k, v, do, causal=causal, window=W, scale=0.3, key_len=kl, o=o)
        for x, y in zip(a, b):
            np.testing.assert_allclose(y, x, atol=1e-11, rtol=0)


def _linear_response_error(lib=None):
    """Largest deviation from the closed-form response of the given-o gradients to a
    change of one element of o: moving o_ic by eps shifts the row sum by eps do_ic,
    hence ds_ij by -p_ij eps do_ic. dq_i moves by -scale eps do_ic sum_j p_ij k_j (the
    forward with k in place of v), dk_j by -scale eps do_ic p_ij q_i (p_ij by brute
    force), every other dq row and all of dv stay."""
    g = torch.Generator().manual_seed(59)
    B, Hq, Hkv, N, d = 1, 2, 1, 23, 8
    q = torch.randn(B, Hq, N, d, generator=g).bfloat16()
    k, v = (torch.randn(B, Hkv, N, d, generator=g).bfloat16() for _ in range(2))
    do = torch.randn(B, Hq, N, d, generator=g).bfloat16()
    scale, eps, (hq, i, c) = 0.4, 1e-3, (1, 9, 5)
    o, _ = oracle.attn_ref(q, k, v, causal=True, scale=scale)
    o2 = o.copy()
    o2[0, hq, i, c] += eps
    dq1, dk1, dv1 = oracle.attn_ref_bwd(q, k, v, do, causal=True, scale=scale, o=o, lib=lib)
    dq2, dk2, dv2 = oracle.attn_ref_bwd(q, k, v, do, causal=True, scale=scale, o=o2, lib=lib)
    pk, _ = oracle.attn_ref(q, k, k, causal=True, scale=scale)
    want = np.zeros_like(dq1)
    want[0, hq, i] = -scale * eps * float(do[0, hq, i, c]) * pk[0, hq, i]
    s = scale * (q[0, hq, i].double() @ k[0, 0].double().T).numpy()
    s[i + 1:] = -np.inf
    p = np.exp(s - s.max())
    p /= p.sum()
    want_k = -scale * eps * float(do[0, hq, i, c]) * p[:, None] * q[0, hq, i].double().numpy()[None, :]
    return max(np.abs(dq2 - dq1 - want).max(), np.abs(dv2 - dv1).max(), np.abs(dk2 - dk1 - want_k[None, None]).max())


def test_bwd_given_o_linear_response():
    assert _linear_response_error() <= 1e-12


GIVEN_O_MUTANTS = {
    # a given output is ignored (the row sum stays the exact one)
    "given_o_ignored": ("for (int64_t c = 0; c < d; ++c) pdp += bf16_bits_to_double(doh[i * d + c]) * oi[c];",
                        "for (int64_t c = 0; c < d; ++c) pdp += p[0] * 0.0 * oi[c];"),
    # a given output read from the wrong row
    "given_o_wrong_row": ("const double *oi = jb->o_in + (bh * N + i) * d;",
                          "const double *oi = jb->o_in + (bh * N + i / 2) * d;"),
}


@pytest.mark.parametrize("name", sorted(GIVEN_O_MUTANTS))
def test_given_o_pin_catches_mutant(name, tmp_path):
    with open(oracle._SRC) as f:
        src = f.read()
    old, new = GIVEN_O_MUTANTS[name]
    assert src.count(old) == 1
    mutated = tmp_path / "attn_ref_mutant.c"
    mutated.write_text(src.replace(old, new))
    so = str(tmp_path / "libattn_ref_mutant.so")
    oracle.build(force=True, src=str(mutated), out=so)
    assert _linear_response_error(oracle.load(so)) > 1e-9, f"mutant {name} not caught"


BWD_MUTANTS = {
    # the softmax gradient without its row term
    "ds_without_row_term": ("const double ds = p[j] * (dp[j] - pdp);", "const double ds = p[j] * dp[j];"),
    # the key gradient without the score scale
    "dk_without_scale": ("dkh[j * d + c] += jb->scale * ds * bf16_bits_to_double(qh[i * d + c]);",
                         "dkh[j * d + c] += ds * bf16_bits_to_double(qh[i * d + c]);"),
    # the value gradient weighted by the score gradient instead of the probability
    "dv_from_ds": ("dvh[j * d + c] += p[j] * bf16_bits_to_double(doh[i * d + c]);",
                   "dvh[j * d + c] += ds * bf16_bits_to_double(doh[i * d + c]);"),
    # the query gradient from value rows instead of key rows
    "dq_from_v": ("dqh[i * d + c] += jb->scale * ds * bf16_bits_to_double(kh[j * d + c]);",
                  "dqh[i * d + c] += jb->scale * ds * bf16_bits_to_double(vh[j * d + c]);"),
}


@pytest.mark.parametrize("name", sorted(BWD_MUTANTS))
def test_bwd_pins_catch_mutant(name, tmp_path):
    with open(oracle._SRC) as f:
        src = f.read()
    old, new = BWD_MUTANTS[name]
    assert src.count(old) == 1
    mutated = tmp_path / "attn_ref_mutant.c"
    mutated.write_text(src.replace(old, new))
    so = str(tmp_path / "libattn_ref_mutant.so")
    oracle.build(force=True, src=str(mutated), out=so)
    lib = oracle.load(so)
    g = torch.Generator().manual_seed(58)
    B, Hq, Hkv, N, d = 1, 2, 1, 12, 8
    q = torch.randn(B, Hq, N, d, generator=g).bfloat16()
    k = torch.randn(B, Hkv, N, d, generator=g).bfloat16()
    v = torch.randn(B, Hkv, N, d, generator=g).bfloat16()
    do = torch.randn(B, Hq, N, d, generator=g).bfloat16()
    dq, dk, dv = oracle.attn_ref_bwd(q, k, v, do, causal=True, scale=0.3, lib=lib)
    qt, kt, vt = (t.double().requires_grad_() for t in (q, k, v))
    o = F.scaled_dot_product_attention(qt, kt.repeat_interleave(2, 1), vt.repeat_interleave(2, 1),
                                       is_causal=True, scale=0.3)
    o.backward(do.double())
    worst = max(np.abs(dq - qt.grad.numpy()).max(), np.abs(dk - kt.grad.numpy()).max(),
                np.abs(dv - vt.grad.numpy()).max())
    assert worst > 1e-6, f"mutant {name} not caught"


def test_dq_rows_match_full_backward():
    # the row-by-row query gradient equals the full backward's, for every row, with and
    # without padding, window and grouped heads
    g = torch.Generator().manual_seed(60)
    B, Hq, Hkv, N, d = 2, 4, 2, 45, 16
    q = torch.randn(B, Hq, N, d, generator=g).bfloat16()
    k, v = (torch.randn(B, Hkv, N, d, generator=g).bfloat16() for _ in range(2))
    do = torch.randn(B, Hq, N, d, generator=g).bfloat16()
    rows = np.arange(B * Hq * N)
    for causal, W, kl in ((True, 0, None), (False, 7, [45, 20]), (True, 11, [30, 45])):
        dq, _, _ = oracle.attn_ref_bwd(q, k, v, do, causal=causal, window=W, scale=0.3, key_len=kl)
        dq_rows = oracle.attn_ref_bwd_dq_rows(q, k, v, do, rows, causal=causal, window=W, scale=0.3, key_len=kl)
        np.testing.assert_allclose(dq_rows, dq.reshape(-1, d), atol=1e-12, rtol=0)
    with pytest.raises(ValueError):
        oracle.attn_ref_bwd_dq_rows(q, k, v, do, [B * Hq * N], causal=True, scale=0.3)


def test_bwd_thread_count_changes_only_rounding():
    # the threads split the query rows into slices whose dk, dv partials are added in
    # slice order: any thread count gives the one-thread gradients up to fp64 rounding,
    # and the same count gives the same bits. Slices here split heads and groups.
    g = torch.Generator().manual_seed(61)
    B, Hq, Hkv, N, d = 2, 4, 2, 41, 16
    q = torch.randn(B, Hq, N, d, generator=g).bfloat16()
    k, v = (torch.randn(B, Hkv, N, d, generator=g).bfloat16() for _ in range(2))
    do = torch.randn(B, Hq, N, d, generator=g).bfloat16()
    one = oracle.attn_ref_bwd(q, k, v, do, causal=True, window=9, scale=0.3, nthreads=1)
    for n in (2, 7, 13, B * Hq * N + 5):
        many = oracle.attn_ref_bwd(q, k, v, do, causal=True, window=9, scale=0.3, nthreads=n)
        again = oracle.attn_ref_bwd(q, k, v, do, causal=True, window=9, scale=0.3, nthreads=n)
        for a, b, c in zip(one, many, again):
            np.testing.assert_allclose(b, a, atol=1e-12, rtol=0)
            assert np.array_equal(b, c)
