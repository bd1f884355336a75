"""Pins for the fp64 oracle: each checks it against something other than itself.

Every pin takes the oracle library handle so the mutation tests can run the same
pins against deliberately broken copies of the oracle. A pin raises AssertionError
on mismatch.

What pins what:
  worked example    the FlashAttention-3 review page's N=4, d=2 inputs, expected values
                    in closed form (dot products of small integers, then exp/log)
  one-hot           N=8, d=4 one-hot rows: every score is 0 or c, so O and LSE have a
                    closed form from residue counts; pins the causal and window masks
  zero query        all scores equal: O is the mean of the visible V rows, LSE = ln |J(i)|
  constant V        O equals that row for any Q, K and mask
  causal row 0      O_0 = V_0 and LSE_0 = scale * q_0 . k_0
  GQA               equals plain multi-head attention on repeat-interleaved K, V
  window >= N       equals plain causal
  permutation       bidirectional O, LSE invariant under a joint permutation of K, V rows
  brute force       mpmath at 40 digits on a small random case (O and LSE)
  library           torch CPU fp64 scaled_dot_product_attention with a boolean mask
  padding           zero-query closed form with per-batch valid lengths (padded rows
                    see nothing); valid rows equal the batch truncated to its length
  symmetric window  one-hot closed form for |i - j| < W; W >= N equals bidirectional;
                    brute force and torch SDPA with padding and both window kinds
  decode shape      queries at the end of a sequence equal the plain forward's last
                    rows; zero-query closed form; brute force and torch SDPA
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def bf16(x) -> torch.Tensor:
    t = torch.as_tensor(np.asarray(x, dtype=np.float32))
    out = t.to(torch.bfloat16)
    assert torch.equal(out.float(), t), "pin inputs must be exact in bf16"
    return out.contiguous()


def f64(t: torch.Tensor) -> np.ndarray:
    return t.double().numpy()


def _close(a, b, tol, what):
    """max |a - b| / max(1, |b|) <= tol; equal infinities match, NaN never does."""
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    if not a.size:
        return
    assert not (np.isnan(a).any() or np.isnan(b).any()), f"{what}: NaN"
    finite = np.isfinite(a) & np.isfinite(b)
    with np.errstate(invalid="ignore", over="ignore"):
        rel = np.abs(a - b) / np.maximum(1.0, np.abs(b))
    err = np.where(a == b, 0.0, np.where(finite, rel, np.inf)).max()
    assert err <= tol, f"{what}: max rel err {err:.3e} > {tol:.1e}"


# ---------------------------------------------------------------- worked example
def pin_worked_example(lib):
    with open(os.path.join(HERE, "golden", "fa3_review_worked_example.json")) as f:
        ex = json.load(f)
    Q, K = ex["Q"], ex["K"]
    for vkey in ("V", "V_alt"):
        V = ex[vkey]
        for scale in (1.0, 1.0 / math.sqrt(2.0)):
            q = bf16(Q).reshape(1, 1, 4, 2)
            k = bf16(K).reshape(1, 1, 4, 2)
            v = bf16(V).reshape(1, 1, 4, 2)
            o, lse = oracle.attn_ref(q, k, v, causal=False, window=0, scale=scale, lib=lib)
            for i in range(4):
                s = [scale * (Q[i][0] * K[j][0] + Q[i][1] * K[j][1]) for j in range(4)]
                m = max(s)
                lse_cf = m + math.log(sum(math.exp(x - m) for x in s))
                p = [math.exp(x - lse_cf) for x in s]
                o_cf = [sum(p[j] * V[j][c] for j in range(4)) for c in range(2)]
                _close(lse[0, 0, i], lse_cf, 1e-13, f"worked example lse row {i}")
                _close(o[0, 0, i], o_cf, 1e-13, f"worked example O row {i}")
    # the specific values quoted in the design notes (unscaled, row 0)
    q = bf16(Q).reshape(1, 1, 4, 2)
    k = bf16(K).reshape(1, 1, 4, 2)
    o, lse = oracle.attn_ref(q, k, bf16(ex["V"]).reshape(1, 1, 4, 2), scale=1.0, lib=lib)
    lse0 = 22.0 + math.log(1.0 + math.exp(-6.0) + math.exp(-12.0) + math.exp(-18.0))
    _close(lse[0, 0, 0], lse0, 1e-14, "row-0 lse closed form")
    assert abs(lse[0, 0, 0] - 22.002482) < 5e-7
    assert abs(o[0, 0, 0, 0] - 0.002473) < 5e-7 and abs(o[0, 0, 0, 1] - 0.002479) < 5e-7
    o, _ = oracle.attn_ref(q, k, bf16(ex["V_alt"]).reshape(1, 1, 4, 2), scale=1.0, lib=lib)
    assert abs(o[0, 0, 0, 0] - 3.997515) < 5e-7
    o, lse = oracle.attn_ref(q, k, bf16(ex["V_alt"]).reshape(1, 1, 4, 2),
                             scale=1.0 / math.sqrt(2.0), lib=lib)
    assert abs(lse[0, 0, 0] - 15.570823) < 5e-7 and abs(o[0, 0, 0, 0] - 3.985421) < 5e-7


# ---------------------------------------------------------------- one-hot closed form
def _count_residue(lo: int, hi: int, r: int, m: int = 4) -> int:
    """#{j in [lo, hi] : j = r (mod m)} for 0 <= lo <= hi + 1."""
    if hi < lo:
        return 0
    return (hi - r) // m - (lo - 1 - r) // m


def pin_one_hot(lib):
    N, d = 8, 4
    a, b = 2.0, 1.5          # exact in bf16
    for scale in (0.5, 1.0 / math.sqrt(d)):
        c = scale * a * b
        q = bf16([[a if col == i % 4 else 0.0 for col in range(d)] for i in range(N)])
        k = bf16([[b if col == j % 4 else 0.0 for col in range(d)] for j in range(N)])
        # v_j = e_{(j+1) mod 4} scaled by 3 - so V is not aligned with K
        v = bf16([[3.0 if col == (j + 1) % 4 else 0.0 for col in range(d)] for j in range(N)])
        cases = [(False, 0), (True, 0), (True, 1), (True, 2), (True, 3), (True, 5), (True, 8)]
        for causal, W in cases:
            o, lse = oracle.attn_ref(q.reshape(1, 1, N, d), k.reshape(1, 1, N, d),
                                     v.reshape(1, 1, N, d), causal=causal, window=W,
                                     scale=scale, lib=lib)
            for i in range(N):
                hi = i if causal else N - 1
                lo = max(0, i - W + 1) if W > 0 else 0
                cnt = [_count_residue(lo, hi, r) for r in range(4)]
                ri = i % 4
                Z = cnt[ri] * math.exp(c) + (sum(cnt) - cnt[ri])
                lse_cf = math.log(Z)
                o_cf = [0.0] * d
                for r in range(4):
                    w = (math.exp(c) if r == ri else 1.0) * cnt[r]
                    o_cf[(r + 1) % 4] += 3.0 * w / Z
                _close(lse[0, 0, i], lse_cf, 1e-13, f"one-hot lse causal={causal} W={W} i={i}")
                _close(o[0, 0, i], o_cf, 1e-13, f"one-hot O causal={causal} W={W} i={i}")


# ---------------------------------------------------------------- zero query
def pin_zero_query(lib):
    g = torch.Generator().manual_seed(11)
    N, d = 37, 8
    q = torch.zeros(1, 2, N, d, dtype=torch.bfloat16)
    k = torch.randn(1, 2, N, d, generator=g).bfloat16()
    v = torch.randn(1, 2, N, d, generator=g).bfloat16()
    vd = f64(v)
    for causal, W in [(False, 0), (True, 0), (True, 1), (True, 4), (True, 16), (True, 100)]:
        o, lse = oracle.attn_ref(q, k, v, causal=causal, window=W, scale=0.3, lib=lib)
        for h in range(2):
            for i in range(N):
                hi = i if causal else N - 1
                lo = max(0, i - W + 1) if W > 0 else 0
                n = hi - lo + 1
                _close(lse[0, h, i], math.log(n), 1e-13, f"zero-q lse W={W} i={i}")
                _close(o[0, h, i], vd[0, h, lo:hi + 1].mean(axis=0), 1e-13, f"zero-q O W={W} i={i}")


# ---------------------------------------------------------------- constant V
def pin_constant_v(lib):
    g = torch.Generator().manual_seed(12)
    B, H, N, d = 2, 2, 29, 16
    q = (3 * torch.randn(B, H, N, d, generator=g)).bfloat16()
    k = torch.randn(B, H, N, d, generator=g).bfloat16()
    row = torch.randn(d, generator=g).bfloat16()
    v = row.expand(B, H, N, d).contiguous()
    for causal, W in [(False, 0), (True, 0), (True, 3)]:
        o, _ = oracle.attn_ref(q, k, v, causal=causal, window=W, scale=0.25, lib=lib)
        _close(o, np.broadcast_to(f64(row), o.shape), 1e-13, f"constant V causal={causal} W={W}")


# ---------------------------------------------------------------- causal first row
def pin_causal_row0(lib):
    g = torch.Generator().manual_seed(13)
    B, H, N, d = 2, 3, 19, 32
    q = torch.randn(B, H, N, d, generator=g).bfloat16()
    k = torch.randn(B, H, N, d, generator=g).bfloat16()
    v = torch.randn(B, H, N, d, generator=g).bfloat16()
    scale = 1.0 / math.sqrt(d)
    for W in (0, 1, 7):
        o, lse = oracle.attn_ref(q, k, v, causal=True, window=W, scale=scale, lib=lib)
        _close(o[:, :, 0], f64(v)[:, :, 0], 1e-14, "causal row 0 O = V_0")
        want = scale * np.einsum("bhc,bhc->bh", f64(q)[:, :, 0], f64(k)[:, :, 0])
        _close(lse[:, :, 0], want, 1e-13, "causal row 0 lse")
    # window 1: every row sees only itself
    o, lse = oracle.attn_ref(q, k, v, causal=True, window=1, scale=scale, lib=lib)
    _close(o, f64(v), 1e-14, "window 1: O = V")
    _close(lse, scale * np.einsum("bhnc,bhnc->bhn", f64(q), f64(k)), 1e-13, "window 1 lse")


# ---------------------------------------------------------------- GQA
def pin_gqa(lib):
    g = torch.Generator().manual_seed(14)
    B, Hkv, G, N, d = 2, 3, 4, 23, 16
    q = torch.randn(B, Hkv * G, N, d, generator=g).bfloat16()
    k = torch.randn(B, Hkv, N, d, generator=g).bfloat16()
    v = torch.randn(B, Hkv, N, d, generator=g).bfloat16()
    kr = k.repeat_interleave(G, dim=1).contiguous()
    vr = v.repeat_interleave(G, dim=1).contiguous()
    for causal, W in [(False, 0), (True, 0), (True, 5)]:
        o1, l1 = oracle.attn_ref(q, k, v, causal=causal, window=W, scale=0.2, lib=lib)
        o2, l2 = oracle.attn_ref(q, kr, vr, causal=causal, window=W, scale=0.2, lib=lib)
        assert np.array_equal(o1, o2) and np.array_equal(l1, l2), "GQA != repeated-KV MHA"


# ---------------------------------------------------------------- window >= N
def pin_window_ge_n(lib):
    g = torch.Generator().manual_seed(15)
    B, H, N, d = 1, 2, 33, 8
    q = torch.randn(B, H, N, d, generator=g).bfloat16()
    k = torch.randn(B, H, N, d, generator=g).bfloat16()
    v = torch.randn(B, H, N, d, generator=g).bfloat16()
    o0, l0 = oracle.attn_ref(q, k, v, causal=True, window=0, scale=0.4, lib=lib)
    for W in (N, N + 1, 10 * N):
        o1, l1 = oracle.attn_ref(q, k, v, causal=True, window=W, scale=0.4, lib=lib)
        assert np.array_equal(o0, o1) and np.array_equal(l0, l1), f"window {W} >= N != causal"
    # and a window smaller than N must differ
    o1, _ = oracle.attn_ref(q, k, v, causal=True, window=N - 1, scale=0.4, lib=lib)
    assert not np.array_equal(o0, o1)


# ---------------------------------------------------------------- permutation
def pin_permutation(lib):
    g = torch.Generator().manual_seed(16)
    B, H, N, d = 1, 2, 31, 16
    q = torch.randn(B, H, N, d, generator=g).bfloat16()
    k = torch.randn(B, H, N, d, generator=g).bfloat16()
    v = torch.randn(B, H, N, d, generator=g).bfloat16()
    perm = torch.randperm(N, generator=g)
    o0, l0 = oracle.attn_ref(q, k, v, scale=0.3, lib=lib)
    o1, l1 = oracle.attn_ref(q, k[:, :, perm].contiguous(), v[:, :, perm].contiguous(),
                             scale=0.3, lib=lib)
    _close(o1, o0, 1e-13, "permutation O")
    _close(l1, l0, 1e-13, "permutation lse")


# ---------------------------------------------------------------- brute force (mpmath)
def pin_brute_force(lib):
    import mpmath
    mpmath.mp.dps = 40
    g = torch.Generator().manual_seed(17)
    B, Hq, Hkv, N, d = 1, 2, 1, 12, 4
    q = (2 * torch.randn(B, Hq, N, d, generator=g)).bfloat16()
    k = (2 * torch.randn(B, Hkv, N, d, generator=g)).bfloat16()
    v = torch.randn(B, Hkv, N, d, generator=g).bfloat16()
    qd, kd, vd = f64(q), f64(k), f64(v)
    scale = 1.0 / math.sqrt(d)
    for causal, W in [(False, 0), (True, 0), (True, 3)]:
        o, lse = oracle.attn_ref(q, k, v, causal=causal, window=W, scale=scale, lib=lib)
        for h in range(Hq):
            for i in range(N):
                js = [j for j in range(N) if (not causal or j <= i) and (W == 0 or i - j < W)]
                s = {j: mpmath.mpf(scale) * mpmath.fsum(mpmath.mpf(qd[0, h, i, c]) * mpmath.mpf(kd[0, 0, j, c])
                                                       for c in range(d)) for j in js}
                z = mpmath.fsum(mpmath.exp(s[j]) for j in js)
                lse_bf = mpmath.log(z)
                o_bf = [mpmath.fsum(mpmath.exp(s[j]) * mpmath.mpf(vd[0, 0, j, c]) for j in js) / z
                        for c in range(d)]
                _close(lse[0, h, i], float(lse_bf), 1e-13, "brute-force lse")
                _close(o[0, h, i], [float(x) for x in o_bf], 1e-13, "brute-force O")


# ---------------------------------------------------------------- library routine
def pin_torch_sdpa(lib):
    import torch.nn.functional as F
    g = torch.Generator().manual_seed(18)
    for (B, Hq, Hkv, N, d) in [(2, 4, 2, 64, 32), (1, 2, 2, 130, 64)]:
        q = torch.randn(B, Hq, N, d, generator=g).bfloat16()
        k = torch.randn(B, Hkv, N, d, generator=g).bfloat16()
        v = torch.randn(B, Hkv, N, d, generator=g).bfloat16()
        G = Hq // Hkv
        q64, k64, v64 = q.double(), k.double().repeat_interleave(G, 1), v.double().repeat_interleave(G, 1)
        scale = 1.0 / math.sqrt(d)
        i = torch.arange(N).view(N, 1)
        j = torch.arange(N).view(1, N)
        for causal, W in [(False, 0), (True, 0), (True, 17)]:
            mask = torch.ones(N, N, dtype=torch.bool)
            if causal:
                mask &= j <= i
            if W:
                mask &= (i - j) < W
            ref = F.scaled_dot_product_attention(q64, k64, v64, attn_mask=mask, scale=scale)
            o, _ = oracle.attn_ref(q, k, v, causal=causal, window=W, scale=scale, lib=lib)
            _close(o, ref.numpy(), 1e-12, f"torch SDPA causal={causal} W={W}")


# ---------------------------------------------------------------- padding and symmetric window
def _visible(i, j, causal, W, L):
    """The mask, restated from the pages for the pins below (right padding to L)."""
    if i >= L or j >= L:
        return False
    if causal and j > i:
        return False
    if W and i - j >= W:
        return False
    if W and not causal and j - i >= W:
        return False
    return True


def pin_padding_zero_query(lib):
    # all scores equal: a valid row averages the V rows it sees, lse = ln(count); a
    # padded row sees nothing (o = 0, lse = -inf)
    g = torch.Generator().manual_seed(21)
    B, N, d = 3, 23, 8
    q = torch.zeros(B, 2, N, d, dtype=torch.bfloat16)
    k = torch.randn(B, 1, N, d, generator=g).bfloat16()
    v = torch.randn(B, 1, N, d, generator=g).bfloat16()
    vd = f64(v)
    key_len = [0, 9, N]
    for causal, W in [(False, 0), (True, 0), (True, 4), (False, 3), (False, 40)]:
        o, lse = oracle.attn_ref(q, k, v, causal=causal, window=W, scale=0.7, lib=lib, key_len=key_len)
        for b in range(B):
            for h in range(2):
                for i in range(N):
                    js = [j for j in range(N) if _visible(i, j, causal, W, key_len[b])]
                    if not js:
                        assert lse[b, h, i] == -np.inf and not o[b, h, i].any(), "padded row"
                        continue
                    _close(lse[b, h, i], math.log(len(js)), 1e-13, f"pad zero-q lse b={b} i={i}")
                    _close(o[b, h, i], vd[b, 0, js].mean(axis=0), 1e-13, f"pad zero-q O b={b} i={i}")


def pin_padding_truncation(lib):
    # the valid rows of a padded batch equal attention over that batch truncated to its
    # valid length, with no padding at all
    g = torch.Generator().manual_seed(22)
    B, Hq, Hkv, N, d = 3, 4, 2, 29, 16
    q = torch.randn(B, Hq, N, d, generator=g).bfloat16()
    k = torch.randn(B, Hkv, N, d, generator=g).bfloat16()
    v = torch.randn(B, Hkv, N, d, generator=g).bfloat16()
    key_len = [29, 1, 17]
    for causal, W in [(False, 0), (True, 0), (True, 5), (False, 6)]:
        o, lse = oracle.attn_ref(q, k, v, causal=causal, window=W, scale=0.3, lib=lib, key_len=key_len)
        for b, L in enumerate(key_len):
            ot, lt = oracle.attn_ref(q[b:b + 1, :, :L].contiguous(), k[b:b + 1, :, :L].contiguous(),
                                     v[b:b + 1, :, :L].contiguous(), causal=causal, window=W, scale=0.3,
                                     lib=lib)
            _close(o[b, :, :L], ot[0], 1e-13, f"truncation O b={b}")
            _close(lse[b, :, :L], lt[0], 1e-13, f"truncation lse b={b}")
            assert np.all(lse[b, :, L:] == -np.inf) and not o[b, :, L:].any()


def pin_symmetric_window_one_hot(lib):
    # the one-hot closed form with a symmetric window: row i sees keys
    # max(0, i-W+1) .. min(N-1, i+W-1)
    N, d = 8, 4
    a, bb = 2.0, 1.5
    scale = 0.5
    c = scale * a * bb
    q = bf16([[a if col == i % 4 else 0.0 for col in range(d)] for i in range(N)])
    k = bf16([[bb if col == j % 4 else 0.0 for col in range(d)] for j in range(N)])
    v = bf16([[3.0 if col == (j + 1) % 4 else 0.0 for col in range(d)] for j in range(N)])
    for W in (1, 2, 3, 5, 8, 20):
        o, lse = oracle.attn_ref(q.reshape(1, 1, N, d), k.reshape(1, 1, N, d), v.reshape(1, 1, N, d),
                                 causal=False, window=W, scale=scale, lib=lib)
        for i in range(N):
            lo, hi = max(0, i - W + 1), min(N - 1, i + W - 1)
            cnt = [_count_residue(lo, hi, r) for r in range(4)]
            ri = i % 4
            Z = cnt[ri] * math.exp(c) + (sum(cnt) - cnt[ri])
            o_cf = [0.0] * d
            for r in range(4):
                w = (math.exp(c) if r == ri else 1.0) * cnt[r]
                o_cf[(r + 1) % 4] += 3.0 * w / Z
            _close(lse[0, 0, i], math.log(Z), 1e-13, f"sym one-hot lse W={W} i={i}")
            _close(o[0, 0, i], o_cf, 1e-13, f"sym one-hot O W={W} i={i}")


def pin_symmetric_window_ge_n(lib):
    g = torch.Generator().manual_seed(23)
    q = torch.randn(1, 2, 31, 8, generator=g).bfloat16()
    k = torch.randn(1, 2, 31, 8, generator=g).bfloat16()
    v = torch.randn(1, 2, 31, 8, generator=g).bfloat16()
    o0, l0 = oracle.attn_ref(q, k, v, scale=0.4, lib=lib)
    for W in (31, 32, 500):
        o1, l1 = oracle.attn_ref(q, k, v, causal=False, window=W, scale=0.4, lib=lib)
        assert np.array_equal(o0, o1) and np.array_equal(l0, l1), f"symmetric window {W} >= N"
    o1, _ = oracle.attn_ref(q, k, v, causal=False, window=30, scale=0.4, lib=lib)
    assert not np.array_equal(o0, o1)


def pin_masks_brute_force(lib):
    import mpmath
    mpmath.mp.dps = 40
    g = torch.Generator().manual_seed(24)
    B, Hq, Hkv, N, d = 2, 2, 1, 11, 4
    q = (2 * torch.randn(B, Hq, N, d, generator=g)).bfloat16()
    k = (2 * torch.randn(B, Hkv, N, d, generator=g)).bfloat16()
    v = torch.randn(B, Hkv, N, d, generator=g).bfloat16()
    qd, kd, vd = f64(q), f64(k), f64(v)
    scale = 0.5
    key_len = [7, 11]
    for causal, W in [(False, 3), (True, 2), (False, 0)]:
        o, lse = oracle.attn_ref(q, k, v, causal=causal, window=W, scale=scale, lib=lib, key_len=key_len)
        for b in range(B):
            for h in range(Hq):
                for i in range(N):
                    js = [j for j in range(N) if _visible(i, j, causal, W, key_len[b])]
                    if not js:
                        assert lse[b, h, i] == -np.inf
                        continue
                    s = {j: mpmath.mpf(scale) * mpmath.fsum(mpmath.mpf(qd[b, h, i, cc]) * mpmath.mpf(kd[b, 0, j, cc])
                                                           for cc in range(d)) for j in js}
                    z = mpmath.fsum(mpmath.exp(s[j]) for j in js)
                    _close(lse[b, h, i], float(mpmath.log(z)), 1e-13, "masks brute-force lse")
                    ob = [float(mpmath.fsum(mpmath.exp(s[j]) * mpmath.mpf(vd[b, 0, j, cc]) for j in js) / z)
                          for cc in range(d)]
                    _close(o[b, h, i], ob, 1e-13, "masks brute-force O")


def pin_masks_torch_sdpa(lib):
    import torch.nn.functional as F
    g = torch.Generator().manual_seed(25)
    B, H, N, d = 2, 2, 70, 32
    q = torch.randn(B, H, N, d, generator=g).bfloat16()
    k = torch.randn(B, H, N, d, generator=g).bfloat16()
    v = torch.randn(B, H, N, d, generator=g).bfloat16()
    key_len = [70, 45]
    i = torch.arange(N).view(N, 1)
    j = torch.arange(N).view(1, N)
    for causal, W in [(False, 9), (False, 0), (True, 13)]:
        o, _ = oracle.attn_ref(q, k, v, causal=causal, window=W, scale=0.2, lib=lib, key_len=key_len)
        for b, L in enumerate(key_len):
            mask = (i < L) & (j < L)
            if causal:
                mask &= j <= i
            if W:
                mask &= (i - j) < W
                if not causal:
                    mask &= (j - i) < W
            ref = F.scaled_dot_product_attention(q[b:b + 1].double(), k[b:b + 1].double(), v[b:b + 1].double(),
                                                 attn_mask=mask, scale=0.2)
            _close(o[b, :, :L], ref[0, :, :L].numpy(), 1e-12, f"torch SDPA masks b={b} c={causal} W={W}")


# ---------------------------------------------------------------- decode shape
def pin_decode_equals_last_rows(lib):
    # Nq queries at the end of an Nk-token sequence are the last Nq rows of the plain
    # forward over all Nk tokens
    g = torch.Generator().manual_seed(31)
    B, Hq, Hkv, Nk, d = 2, 4, 2, 37, 16
    q = torch.randn(B, Hq, Nk, d, generator=g).bfloat16()
    k = torch.randn(B, Hkv, Nk, d, generator=g).bfloat16()
    v = torch.randn(B, Hkv, Nk, d, generator=g).bfloat16()
    for causal, W in [(True, 0), (True, 5), (False, 0), (False, 7)]:
        of, lf = oracle.attn_ref(q, k, v, causal=causal, window=W, scale=0.3, lib=lib)
        for Nq in (1, 3, 37):
            od, ld = oracle.attn_ref_decode(q[:, :, Nk - Nq:].contiguous(), k, v, causal=causal,
                                            window=W, scale=0.3, lib=lib)
            assert np.array_equal(od, of[:, :, Nk - Nq:]) and np.array_equal(ld, lf[:, :, Nk - Nq:]), \
                f"decode != last rows (causal={causal} W={W} Nq={Nq})"


def pin_decode_zero_query(lib):
    g = torch.Generator().manual_seed(32)
    B, Nq, Nk, d = 1, 3, 20, 8
    q = torch.zeros(B, 2, Nq, d, dtype=torch.bfloat16)
    k = torch.randn(B, 1, Nk, d, generator=g).bfloat16()
    v = torch.randn(B, 1, Nk, d, generator=g).bfloat16()
    vd = f64(v)
    for causal, W in [(True, 0), (True, 4), (False, 0)]:
        o, lse = oracle.attn_ref_decode(q, k, v, causal=causal, window=W, scale=0.5, lib=lib)
        for i in range(Nq):
            pos = Nk - Nq + i
            js = [j for j in range(Nk) if _visible(pos, j, causal, W, Nk)]
            for h in range(2):
                _close(lse[0, h, i], math.log(len(js)), 1e-13, "decode zero-q lse")
                _close(o[0, h, i], vd[0, 0, js].mean(axis=0), 1e-13, "decode zero-q O")


def pin_decode_brute_force_and_sdpa(lib):
    import mpmath
    import torch.nn.functional as F
    mpmath.mp.dps = 40
    g = torch.Generator().manual_seed(33)
    B, Hq, Hkv, Nq, Nk, d = 1, 4, 1, 2, 13, 4
    q = (2 * torch.randn(B, Hq, Nq, d, generator=g)).bfloat16()
    k = (2 * torch.randn(B, Hkv, Nk, d, generator=g)).bfloat16()
    v = torch.randn(B, Hkv, Nk, d, generator=g).bfloat16()
    qd, kd, vd = f64(q), f64(k), f64(v)
    for causal, W in [(True, 0), (True, 6)]:
        o, lse = oracle.attn_ref_decode(q, k, v, causal=causal, window=W, scale=0.5, lib=lib)
        for h in range(Hq):
            for i in range(Nq):
                pos = Nk - Nq + i
                js = [j for j in range(Nk) if _visible(pos, j, causal, W, Nk)]
                s = {j: mpmath.mpf(0.5) * mpmath.fsum(mpmath.mpf(qd[0, h, i, c]) * mpmath.mpf(kd[0, 0, j, c])
                                                     for c in range(d)) for j in js}
                z = mpmath.fsum(mpmath.exp(s[j]) for j in js)
                _close(lse[0, h, i], float(mpmath.log(z)), 1e-13, "decode brute-force lse")
                ob = [float(mpmath.fsum(mpmath.exp(s[j]) * mpmath.mpf(vd[0, 0, j, c]) for j in js) / z)
                      for c in range(d)]
                _close(o[0, h, i], ob, 1e-13, "decode brute-force O")
        i = torch.arange(Nq).view(Nq, 1) + (Nk - Nq)
        j = torch.arange(Nk).view(1, Nk)
        mask = (j <= i) & ((i - j) < W if W else torch.ones(Nq, Nk, dtype=torch.bool))
        ref = F.scaled_dot_product_attention(q.double(), k.double().repeat_interleave(Hq, 1),
                                             v.double().repeat_interleave(Hq, 1), attn_mask=mask, scale=0.5)
        _close(o, ref.numpy(), 1e-12, "decode torch SDPA")


ALL_PINS = [pin_worked_example, pin_one_hot, pin_zero_query, pin_constant_v, pin_causal_row0,
            pin_gqa, pin_window_ge_n, pin_permutation, pin_brute_force, pin_torch_sdpa,
            pin_padding_zero_query, pin_padding_truncation, pin_symmetric_window_one_hot,
            pin_symmetric_window_ge_n, pin_masks_brute_force, pin_masks_torch_sdpa,
            pin_decode_equals_last_rows, pin_decode_zero_query, pin_decode_brute_force_and_sdpa]
