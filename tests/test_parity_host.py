"""The element-by-element comparator used by the GPU parity tests, checked on CPU:
it accepts the oracle's own values rounded to the bf16 output format and rejects
planted errors in O and in the LSE."""
import numpy as np
import pytest
import torch

from parity import compare


def _case(seed=0, n=4096):
    rng = np.random.default_rng(seed)
    o_ref = rng.normal(size=(n, 64)) * 0.3
    lse_ref = rng.normal(size=(n,)) * 3
    return o_ref, lse_ref


def _as_gpu(o, lse):
    return torch.from_numpy(o).float().to(torch.bfloat16), torch.from_numpy(lse).float()


def test_accepts_oracle_rounded_to_output_format():
    o_ref, lse_ref = _case()
    stats = compare(*_as_gpu(o_ref, lse_ref), o_ref, lse_ref, "rounded")
    assert stats["o_max_abs"] <= 2 ** -8 and stats["format_floor_exceptions"] == 0


def test_rejects_one_bad_element():
    o_ref, lse_ref = _case(1)
    o = o_ref.copy()
    o[17, 5] += 0.03
    with pytest.raises(AssertionError, match="exceed"):
        compare(*_as_gpu(o, lse_ref), o_ref, lse_ref, "planted")


def test_rejects_biased_output():
    o_ref, lse_ref = _case(2)
    with pytest.raises(AssertionError, match="mean"):
        compare(*_as_gpu(o_ref + 0.004, lse_ref), o_ref, lse_ref, "biased")


def test_rejects_lse_error():
    o_ref, lse_ref = _case(3)
    lse = lse_ref.copy()
    lse[3] = lse_ref[3] + 2e-3 * max(1.0, abs(lse_ref[3]))
    with pytest.raises(AssertionError, match="LSE"):
        compare(*_as_gpu(o_ref, lse), o_ref, lse_ref, "lse")


def test_format_floor_exception_only_for_large_outputs():
    o_ref, lse_ref = _case(4)
    o_ref[0, 0] = 5.015  # bf16 spacing at 5 is 2^-5: rounding alone can exceed 1e-2
    o = o_ref.copy()
    o[0, 0] = 5.0
    stats = compare(*_as_gpu(o, lse_ref), o_ref, lse_ref, "floor")
    assert stats["o_max_abs"] > 1e-2 and stats["format_floor_exceptions"] == 1


def test_strict_bar_has_no_floor_and_no_exceptions():
    # an fp32 output is held to the plain bar: the element that the bf16 format floor
    # excuses above fails, and so does a mean error inside the floor allowance
    o_ref, lse_ref = _case(5)
    o_ref[0, 0] = 5.015
    o = o_ref.copy()
    o[0, 0] = 5.0
    with pytest.raises(AssertionError, match="strict"):
        compare(torch.from_numpy(o).float(), torch.from_numpy(lse_ref).float(), o_ref, lse_ref, "strict",
                strict=True)
    o_ref, lse_ref = _case(6, n=8)
    o = o_ref + 1.5e-3
    with pytest.raises(AssertionError, match="mean"):
        compare(torch.from_numpy(o).float(), torch.from_numpy(lse_ref).float(), o_ref, lse_ref, "strict mean",
                strict=True)
    stats = compare(torch.from_numpy(o_ref).float(), torch.from_numpy(lse_ref).float(), o_ref, lse_ref,
                    "exact", strict=True)
    assert stats["o_max_abs"] < 1e-6 and stats["format_floor_exceptions"] == 0
