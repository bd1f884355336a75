"""The oracle against what the pages and the mathematics fix (CPU only)."""
import numpy as np
import pytest
import torch

import oracle
import oracle_pins as P


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("pin", P.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin, lib):
    pin(lib)


def test_rows_subset_matches_full(lib):
    g = torch.Generator().manual_seed(3)
    q = torch.randn(2, 4, 45, 16, generator=g).bfloat16()
    k = torch.randn(2, 2, 45, 16, generator=g).bfloat16()
    v = torch.randn(2, 2, 45, 16, generator=g).bfloat16()
    o, lse = oracle.attn_ref(q, k, v, causal=True, window=9, scale=0.25, lib=lib)
    rows = np.array([0, 5, 44, 45, 2 * 4 * 45 - 1, 200], dtype=np.int64)
    o_r, l_r = oracle.attn_ref_rows(q, k, v, True, 9, 0.25, rows, nthreads=3, lib=lib)
    assert np.array_equal(o_r, o.reshape(-1, 16)[rows])
    assert np.array_equal(l_r, lse.reshape(-1)[rows])


def test_thread_count_does_not_change_result(lib):
    g = torch.Generator().manual_seed(4)
    q = torch.randn(1, 2, 70, 8, generator=g).bfloat16()
    k = torch.randn(1, 2, 70, 8, generator=g).bfloat16()
    v = torch.randn(1, 2, 70, 8, generator=g).bfloat16()
    a = oracle.attn_ref(q, k, v, causal=True, scale=0.3, nthreads=1, lib=lib)
    b = oracle.attn_ref(q, k, v, causal=True, scale=0.3, nthreads=7, lib=lib)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("bad", [
    dict(window=-1, causal=True), dict(scale=0.0), dict(scale=float("nan")),
])
def test_rejects_bad_arguments(lib, bad):
    q = torch.zeros(1, 1, 4, 8, dtype=torch.bfloat16)
    kw = dict(causal=False, window=0, scale=0.5)
    kw.update(bad)
    with pytest.raises(ValueError):
        oracle.attn_ref_rows(q, q, q, kw["causal"], kw["window"], kw["scale"], lib=lib)


def test_rejects_bad_group(lib):
    q = torch.zeros(1, 3, 4, 8, dtype=torch.bfloat16)
    k = torch.zeros(1, 2, 4, 8, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        oracle.attn_ref_rows(q, k, k, False, 0, 0.5, lib=lib)
