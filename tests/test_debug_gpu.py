"""The index-checked debug build (libattn_fwd_debug.so, compiled with ATTN_DEBUG).

Its kernels check, before each access, the indices the scheduling arithmetic produces
(shared-memory stages and buffers, tensor-memory column ranges, tensor-map coordinates,
global rows written, per-batch lengths and per-block scales read). A failed check skips
the access and sets a status bit instead of faulting. This stands in for a memory
checker: every entry point runs on the test shapes (ragged tails, grouped heads,
windows, padding, the decode shape with and without splits, e4m3 operands, the
backward) through both builds, the results must be the release build's bits, and no
check may fail. A self-test kernel fails one check on purpose (site 99, no access) to
show that a failure is reported.
"""
from __future__ import annotations

import ctypes
import math
import os

import pytest
import torch

import exact_self_attention_fwd_b300 as ea
from exact_self_attention_fwd_b300.inputs import make_dout, make_qkv, make_qkv_decode, make_signs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def dbg():
    if not os.path.exists(ea.DEBUG_LIB_PATH):
        pytest.fail("libattn_fwd_debug.so is missing: build it with "
                    "`python -m exact_self_attention_fwd_b300.build --debug`")
    lib = ea.load(ea.DEBUG_LIB_PATH)
    lib.attn_device_error(1)
    lib.attn_debug_first_site(1)
    return lib


def clean(lib):
    status = lib.attn_device_error(1)
    site = lib.attn_debug_first_site(1)
    assert status == ea.ATTN_OK and site == 0, f"debug build: status {status}, first failed check {site}"


def both(dbg, fn):
    """fn() under the release build, then under the debug build; results as lists."""
    rel = [t.clone() for t in fn()]
    torch.cuda.synchronize()
    with ea.using(dbg):
        deb = [t.clone() for t in fn()]
    torch.cuda.synchronize()
    clean(dbg)
    for a, b in zip(rel, deb):
        assert torch.equal(a, b), "the debug build changed a result"
    return rel


def test_build_flags(dbg):
    assert dbg.attn_debug_build() == 1
    assert ea.load().attn_debug_build() == 0
    assert ea.load().attn_debug_selftest() == ea.ATTN_ERR_UNSUPPORTED


def test_failed_check_is_reported(dbg):
    assert dbg.attn_debug_selftest() == ea.ATTN_OK
    assert dbg.attn_device_error(1) == ea.ATTN_ERR_BOUNDS
    assert dbg.attn_debug_first_site(1) == 99
    assert dbg.attn_device_error(1) == ea.ATTN_OK and dbg.attn_debug_first_site(1) == 0


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal,W", [(False, 0), (True, 0), (True, 100), (False, 77)])
@pytest.mark.parametrize("N", [1, 127, 129, 300])
def test_forward(dbg, N, d, causal, W):
    q, k, v = (t.to(DEV) for t in make_qkv(2, 4, 2, N, d, 7000 + N + d))
    both(dbg, lambda: ea.attn_fwd(q, k, v, causal=causal, window=W))
    both(dbg, lambda: ea.attn_fwd(q, k, v, causal=causal, window=W, out_fp32=True))


def test_forward_gqa_padding_many_units(dbg):
    q, k, v = (t.to(DEV) for t in make_qkv(5, 16, 2, 700, 128, 7100))
    kl = torch.tensor([0, 1, 129, 500, 700], dtype=torch.int32, device=DEV)
    both(dbg, lambda: ea.attn_fwd(q, k, v, causal=True, key_len=kl))
    both(dbg, lambda: ea.attn_fwd(q, k, v, causal=False, window=64, key_len=kl))
    q, k, v = (t.to(DEV) for t in make_qkv(4, 40, 8, 520, 64, 7101))
    both(dbg, lambda: ea.attn_fwd(q, k, v, causal=True))


@pytest.mark.parametrize("splits", [1, 3, 0])
def test_decode(dbg, splits):
    q, k, v = (t.to(DEV) for t in make_qkv_decode(2, 16, 2, 4, 3000, 128, 7200 + splits))
    both(dbg, lambda: ea.attn_fwd_decode(q, k, v, causal=True, window=500, splits=splits))
    q, k, v = (t.to(DEV) for t in make_qkv_decode(4, 32, 8, 1, 1000, 64, 7210 + splits))
    both(dbg, lambda: ea.attn_fwd_decode(q, k, v, causal=True, splits=splits))


def test_decode_noalloc(dbg):
    q, k, v = (t.to(DEV) for t in make_qkv_decode(4, 32, 8, 1, 4096, 128, 7300))
    B, Hq, Nq, d = q.shape

    def run():
        o = torch.empty_like(q)
        lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=DEV)
        rc = ea.load().attn_fwd_decode_noalloc(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, Hq, k.shape[1], Nq,
            k.shape[2], d, 1, 0, ctypes.c_float(1 / math.sqrt(d)), 0,
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert rc == ea.ATTN_OK
        return o, lse

    both(dbg, run)


def test_fp8_and_quantisers(dbg):
    q, k, v = (t.to(DEV) for t in make_qkv(2, 8, 2, 300, 128, 7400))
    signs = make_signs(128, 7401)
    both(dbg, lambda: ea.quantize_e4m3(q))
    both(dbg, lambda: ea.quantize_e4m3_hadamard(k, signs))
    (q8, qs), (k8, ks), (v8, vs) = (ea.quantize_e4m3(t) for t in (q, k, v))
    both(dbg, lambda: ea.attn_fwd_fp8(q8, k8, v8, qs, ks, vs, causal=True))


@pytest.mark.parametrize("case", [(1, 2, 2, 129, 64, True, 0, None), (2, 8, 2, 300, 128, True, 90, [300, 131]),
                                  (1, 4, 1, 520, 64, False, 130, None)])
def test_backward(dbg, case):
    B, Hq, Hkv, N, d, causal, W, kl = case
    q, k, v = (t.to(DEV) for t in make_qkv(B, Hq, Hkv, N, d, 7500 + N))
    do = make_dout(B, Hq, N, d, 7501 + N).to(DEV)
    klt = None if kl is None else torch.tensor(kl, dtype=torch.int32, device=DEV)
    o, lse = ea.attn_fwd(q, k, v, causal=causal, window=W, key_len=klt)
    both(dbg, lambda: ea.attn_bwd(q, k, v, o, lse, do, causal=causal, window=W, key_len=klt))


def test_host_entry(dbg):
    q, k, v = make_qkv(3, 10, 5, 260, 64, 7600)
    keep = []

    def run():
        hq, hk, hv = q.pin_memory(), k.pin_memory(), v.pin_memory()
        keep.extend([hq, hk, hv])
        ho = torch.empty_like(q).pin_memory()
        hl = torch.empty(3, 10, 260, dtype=torch.float32).pin_memory()
        dq, dk, dv = torch.empty_like(q, device=DEV), torch.empty_like(k, device=DEV), torch.empty_like(v, device=DEV)
        ea.attn_fwd_host(hq, hk, hv, ho, hl, dq, dk, dv, torch.empty_like(q, device=DEV),
                         torch.empty(3, 10, 260, dtype=torch.float32, device=DEV), causal=True)
        torch.cuda.synchronize()
        return ho, hl

    both(dbg, run)
