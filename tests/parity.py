"""Element-by-element comparison of the CUDA path with the fp64 oracle.

Tolerances (the stated bar for floating-point parity):
  O    max |O_gpu - O_ref| <= 1e-2 and mean |O_gpu - O_ref| <= 1e-3 + F over the compared
       elements, where F = mean |bf16_rne(O_ref) - O_ref| is the mean error that storing O
       as bf16 forces on its own (about 1e-5 on the benchmark workloads, but about 1e-3
       when a row sees only a few keys and |O| is of order 1); with one reported
       exception class: an element may exceed 1e-2 only if
       |O_ref| >= 4 and O_gpu is within one bf16 ulp of O_ref rounded to bf16. For
       |O| in [4, 8) half a bf16 ulp is 2^-6 = 0.0156 > 1e-2, so the output format alone
       can break the absolute bound there; such elements are counted and returned, not
       silently passed.
  LSE  |lse_gpu - lse_ref| <= 1e-3 * max(1, |lse_ref|)  (relative, read as absolute near 0)

With strict=True (for O written as fp32, where the output format adds nothing) the bar
is the plain one: max <= 1e-2 and mean <= 1e-3, no floor term and no exceptions.
"""
from __future__ import annotations

import numpy as np
import torch

O_MAX_ABS = 1e-2
O_MEAN_ABS = 1e-3
LSE_REL = 1e-3


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    ax = np.maximum(np.abs(x), np.finfo(np.float32).tiny)
    return np.exp2(np.floor(np.log2(ax)) - 7)


def compare(o_gpu, lse_gpu, o_ref, lse_ref, label: str = "", strict: bool = False) -> dict:
    o = o_gpu.detach().float().cpu().double().numpy().reshape(o_ref.shape)
    lse = lse_gpu.detach().float().cpu().double().numpy().reshape(lse_ref.shape)
    assert np.isfinite(o).all(), f"{label}: non-finite O"
    assert np.isfinite(lse).all(), f"{label}: non-finite LSE"
    err = np.abs(o - o_ref)
    over = err > O_MAX_ABS
    n_floor = 0
    if over.any() and strict:
        raise AssertionError(f"{label}: {int(over.sum())} O elements exceed {O_MAX_ABS} "
                             f"(max {err.max():.4g}) under the strict bar")
    if over.any():
        ref_rne = torch.from_numpy(o_ref[over]).float().to(torch.bfloat16).double().numpy()
        floor_ok = (np.abs(o_ref[over]) >= 4.0) & (np.abs(o[over] - ref_rne) <= bf16_ulp(o_ref[over]))
        bad = int((~floor_ok).sum())
        assert bad == 0, (f"{label}: {bad} O elements exceed {O_MAX_ABS} (max {err.max():.4g}) "
                          f"outside the bf16 format floor")
        n_floor = int(floor_ok.sum())
    mean_abs = float(err.mean()) if err.size else 0.0
    rne = torch.from_numpy(np.ascontiguousarray(o_ref)).float().to(torch.bfloat16).double().numpy()
    floor = float(np.abs(rne - o_ref).mean()) if err.size else 0.0
    allowance = 0.0 if strict else floor
    assert mean_abs <= O_MEAN_ABS + allowance, (f"{label}: mean |dO| {mean_abs:.3g} > {O_MEAN_ABS} + "
                                            f"allowance {allowance:.3g}")
    lerr = np.abs(lse - lse_ref) / np.maximum(1.0, np.abs(lse_ref))
    lmax = float(lerr.max()) if lerr.size else 0.0
    assert lmax <= LSE_REL, f"{label}: LSE rel err {lmax:.3g} > {LSE_REL}"
    return {"o_max_abs": float(err.max()) if err.size else 0.0, "o_mean_abs": mean_abs,
            "o_mean_format_floor": floor,
            "lse_max_rel": lmax, "format_floor_exceptions": n_floor}


def sample_rows(B: int, Hq: int, N: int, window: int, n_random: int, seed: int) -> np.ndarray:
    """Flat row ids ((b*Hq)+hq)*N + i: tile edges, the ends, window edges, and random rows,
    over the first, last and some middle (b, hq)."""
    rng = np.random.default_rng(seed)
    special = {0, 1, 2, 63, 64, 126, 127, 128, 129, 255, 256, 257, N // 2, N - 129, N - 128,
               N - 2, N - 1}
    if window:
        special |= {window - 2, window - 1, window, window + 1, window + 127, window + 128}
    special = sorted(i for i in special if 0 <= i < N)
    bhs = sorted({0, B * Hq - 1, (B * Hq) // 2, int(rng.integers(B * Hq))})
    rows = [bh * N + i for bh in bhs for i in special]
    rows += list(rng.integers(0, B * Hq * N, size=n_random))
    return np.unique(np.asarray(rows, dtype=np.int64))
