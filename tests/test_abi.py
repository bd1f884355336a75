"""The C-ABI library loads on a machine without a GPU, exports every entry point the
header declares, and rejects bad arguments on the host before touching CUDA."""
import ctypes
import subprocess

import pytest

import exact_self_attention_fwd_b300 as ea
from exact_self_attention_fwd_b300 import _lib


@pytest.fixture(scope="module")
def lib():
    from exact_self_attention_fwd_b300 import build
    build.build()
    return ea.load()


def test_exports_every_declared_symbol(lib):
    names = ea.header_functions()
    assert set(names) >= {"attn_fwd", "attn_fwd_padded", "attn_fwd_decode",
                          "attn_fwd_decode_workspace_size", "attn_fwd_decode_noalloc",
                          "attn_quantize_e4m3", "attn_fwd_fp8",
                          "attn_fwd_host", "attn_status_str",
                          "attn_last_cuda_error",
                          "attn_device_error", "attn_selftest_wait_timeout", "attn_version"}
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for n in names:
        assert n in exported, f"{n} declared in attn_api.h but not exported"
        assert hasattr(lib, n)


def test_debug_build_exports_every_declared_symbol():
    # the index-checked build is a drop-in replacement: same exported entry points
    from exact_self_attention_fwd_b300 import build
    build.build(debug=True)
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.DEBUG_LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for n in ea.header_functions():
        assert n in exported, f"{n} declared in attn_api.h but not exported by the debug build"
    dbg = ea.load(_lib.DEBUG_LIB_PATH)
    assert dbg.attn_debug_build() == 1 and ea.load().attn_debug_build() == 0


def test_status_strings(lib):
    for code in range(-9, 1):
        s = lib.attn_status_str(code).decode()
        assert s.startswith("ATTN_")
    assert lib.attn_status_str(-99).decode() == "unknown attn_status"
    assert lib.attn_version() >= 100


A = 1 << 20  # a fake, 16-byte aligned "device address": never dereferenced by these calls


def call(lib, q=A, k=A, v=A, o=A, lse=A, B=1, Hq=1, Hkv=1, N=128, d=64, causal=0, window=0,
         scale=0.125):
    return lib.attn_fwd(q, k, v, o, lse, B, Hq, Hkv, N, d, causal, window, scale, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), ea.ATTN_ERR_NULLPTR),
    (dict(lse=None), ea.ATTN_ERR_NULLPTR),
    (dict(B=0), ea.ATTN_ERR_SHAPE),
    (dict(N=0), ea.ATTN_ERR_SHAPE),
    (dict(Hq=3, Hkv=2), ea.ATTN_ERR_SHAPE),
    (dict(window=-1, causal=1), ea.ATTN_ERR_SHAPE),
    (dict(scale=0.0), ea.ATTN_ERR_SHAPE),
    (dict(scale=float("inf")), ea.ATTN_ERR_SHAPE),
    (dict(scale=float("nan")), ea.ATTN_ERR_SHAPE),
    (dict(causal=2), ea.ATTN_ERR_SHAPE),
    (dict(d=96), ea.ATTN_ERR_UNSUPPORTED),
    (dict(d=256), ea.ATTN_ERR_UNSUPPORTED),
    (dict(q=A + 8), ea.ATTN_ERR_ALIGN),
    (dict(o=A + 2), ea.ATTN_ERR_ALIGN),
    (dict(lse=A + 2), ea.ATTN_ERR_ALIGN),
    (dict(N=(1 << 30) + 1), ea.ATTN_ERR_SHAPE),
    (dict(B=1 << 16, Hq=1 << 16, Hkv=1 << 16), ea.ATTN_ERR_SHAPE),
])
def test_rejects_bad_arguments_before_launch(lib, kw, code):
    assert call(lib, **kw) == code


def test_padded_entry_validates_key_len(lib):
    args = [A] * 5
    assert lib.attn_fwd_padded(*args, None, 1, 1, 1, 128, 64, 0, 0, 0.125, None) == ea.ATTN_ERR_NULLPTR
    assert lib.attn_fwd_padded(*args, A + 2, 1, 1, 1, 128, 64, 0, 0, 0.125, None) == ea.ATTN_ERR_ALIGN
    assert lib.attn_fwd_padded(*args, A, 1, 1, 1, 128, 96, 0, 0, 0.125, None) == ea.ATTN_ERR_UNSUPPORTED


def dcall(lib, q=A, k=A, v=A, o=A, lse=A, B=1, Hq=4, Hkv=1, Nq=1, Nk=256, d=128, causal=1,
          window=0, scale=0.1, splits=1, ws=None, ws_bytes=0):
    return lib.attn_fwd_decode(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, causal, window, scale, splits,
                               ws, ws_bytes, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), ea.ATTN_ERR_NULLPTR),
    (dict(Nq=0), ea.ATTN_ERR_SHAPE),
    (dict(Nq=300, Nk=299), ea.ATTN_ERR_SHAPE),          # more queries than keys
    (dict(Hq=6, Hkv=4), ea.ATTN_ERR_SHAPE),
    (dict(Hq=64, Hkv=1, Nq=4), ea.ATTN_ERR_UNSUPPORTED),  # 256 packed rows > one tile
    (dict(d=96), ea.ATTN_ERR_UNSUPPORTED),
    (dict(window=-2), ea.ATTN_ERR_SHAPE),
    (dict(o=A + 8), ea.ATTN_ERR_ALIGN),
])
def test_decode_rejects_bad_arguments(lib, kw, code):
    assert dcall(lib, **kw) == code


def test_decode_workspace_size(lib):
    # one split needs none; otherwise splits x rows x (d fp32 + 1 fp32 LSE), O part
    # padded to 256 bytes
    assert lib.attn_fwd_decode_workspace_size(2, 8, 2, 3, 1000, 128, 1) == 0
    rows = 2 * 2 * 4 * 3
    o_bytes = 5 * rows * 128 * 4
    assert lib.attn_fwd_decode_workspace_size(2, 8, 2, 3, 1000, 128, 5) == \
        (o_bytes + 255) // 256 * 256 + 5 * rows * 4
    # a split count above the number of 128-key tiles is reduced to it (8 tiles here)
    assert lib.attn_fwd_decode_workspace_size(1, 4, 1, 1, 1000, 64, 50) == \
        lib.attn_fwd_decode_workspace_size(1, 4, 1, 1, 1000, 64, 8)
    assert lib.attn_fwd_decode_workspace_size(1, 4, 3, 1, 100, 64, 2) == 0   # bad shape


def test_fp8_entries_validate(lib):
    assert lib.attn_quantize_e4m3(None, A, A, 1, 128, 128, None) == ea.ATTN_ERR_NULLPTR
    assert lib.attn_quantize_e4m3(A, A, A, 1, 128, 96, None) == ea.ATTN_ERR_UNSUPPORTED
    assert lib.attn_quantize_e4m3(A, A + 4, A, 1, 128, 128, None) == ea.ATTN_ERR_ALIGN
    assert lib.attn_quantize_e4m3(A, A, A, 70000, 128, 128, None) == ea.ATTN_ERR_SHAPE
    args = [A, A, A, A, A, A, A, A, 1, 1, 1, 128]
    assert lib.attn_fwd_fp8(*args, 64, 0, 0, 0.1, None) == ea.ATTN_ERR_UNSUPPORTED
    bad = list(args)
    bad[3] = None
    assert lib.attn_fwd_fp8(*bad, 128, 0, 0, 0.1, None) == ea.ATTN_ERR_NULLPTR
    bad = list(args)
    bad[4] = A + 2
    assert lib.attn_fwd_fp8(*bad, 128, 0, 0, 0.1, None) == ea.ATTN_ERR_ALIGN


def test_host_entry_validates_both_buffer_sets(lib):
    args = [A] * 10 + [1, 1, 1, 128, 64, 0, 0, 0.125, None]
    bad = list(args)
    bad[0] = None
    assert lib.attn_fwd_host(*bad) == ea.ATTN_ERR_NULLPTR
    bad = list(args)
    bad[9] = A + 1
    assert lib.attn_fwd_host(*bad) == ea.ATTN_ERR_ALIGN


def test_selftest_rejects_bad_limit(lib):
    assert lib.attn_selftest_wait_timeout(0) == ea.ATTN_ERR_SHAPE
    assert lib.attn_selftest_wait_timeout(2_000_000_000) == ea.ATTN_ERR_SHAPE


def test_valid_call_without_gpu_reports_cuda_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; covered by the GPU tests")
    assert call(lib) == ea.ATTN_ERR_CUDA
    assert lib.attn_last_cuda_error() != 0


def test_python_binding_refuses_cpu_tensors(lib):
    import torch
    q = torch.zeros(1, 1, 128, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        ea.attn_fwd(q, q, q)


def test_sign_masks():
    signs = [1.0] * 128
    assert ea.sign_masks(signs) == (0, 0)
    signs[0] = signs[63] = signs[64] = signs[127] = -1.0
    assert ea.sign_masks(signs) == ((1 << 63) | 1, (1 << 63) | 1)
    with pytest.raises(ValueError):
        ea.sign_masks([1.0] * 127)
    with pytest.raises(ValueError):
        ea.sign_masks([0.5] * 128)


def test_backward_entry_validates(lib):
    # q, k, v, o, lse, dout, dq, dk, dv, key_len, B, Hq, Hkv, N, d, causal, window, scale,
    # workspace, workspace_bytes, stream
    need = lib.attn_bwd_workspace_size(1, 2, 300, 128)
    # (lse log2(e), D) per row, rows padded to 384
    assert need == 2 * 1 * 2 * 384 * 4
    assert lib.attn_bwd_workspace_size(1, 2, 300, 96) == 0
    args = [A] * 9 + [None, 1, 2, 1, 300, 128, 1, 0, 0.1, A, need, None]
    for i in (0, 5, 6, 7, 8, 18):
        bad = list(args)
        bad[i] = None
        assert lib.attn_bwd(*bad) == ea.ATTN_ERR_NULLPTR, i
    bad = list(args)
    bad[14] = 96
    assert lib.attn_bwd(*bad) == ea.ATTN_ERR_UNSUPPORTED
    bad = list(args)
    bad[12] = 3                                   # Hq not a multiple of Hkv
    assert lib.attn_bwd(*bad) == ea.ATTN_ERR_SHAPE
    bad = list(args)
    bad[6] = A + 8                                # dq not 16-byte aligned
    assert lib.attn_bwd(*bad) == ea.ATTN_ERR_ALIGN
    bad = list(args)
    bad[18] = A + 16                              # workspace not 256-byte aligned
    assert lib.attn_bwd(*bad) == ea.ATTN_ERR_ALIGN
    bad = list(args)
    bad[19] = need - 4
    assert lib.attn_bwd(*bad) == ea.ATTN_ERR_WORKSPACE


def test_hadamard_quantiser_validates(lib):
    assert lib.attn_quantize_e4m3_hadamard(None, 0, 0, A, A, 1, 128, 128, None) == ea.ATTN_ERR_NULLPTR
    assert lib.attn_quantize_e4m3_hadamard(A, 0, 0, A, A, 1, 128, 64, None) == ea.ATTN_ERR_UNSUPPORTED
    assert lib.attn_quantize_e4m3_hadamard(A, 0, 0, A + 8, A, 1, 128, 128, None) == ea.ATTN_ERR_ALIGN
    assert lib.attn_quantize_e4m3_hadamard(A, 0, 0, A, A, 70000, 128, 128, None) == ea.ATTN_ERR_SHAPE
