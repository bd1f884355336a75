"""ctypes binding of libattn_fwd.so: argument marshalling only.

Every step of the attention computation runs in the CUDA library. There is no CPU
or PyTorch fallback: if the library is missing this module raises, and every call
refuses tensors that are not CUDA bf16/fp32 of the required shape.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import re

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
LIB_PATH = os.path.join(PKG, "libattn_fwd.so")
HEADER = os.path.join(ROOT, "include", "attn_api.h")

ATTN_OK = 0
ATTN_ERR_NULLPTR = -1
ATTN_ERR_ALIGN = -2
ATTN_ERR_SHAPE = -3
ATTN_ERR_UNSUPPORTED = -4
ATTN_ERR_CUDA = -5
ATTN_ERR_TIMEOUT = -6
ATTN_ERR_WORKSPACE = -7
ATTN_ERR_SCRATCH_LIMIT = -8
ATTN_ERR_BOUNDS = -9
DEBUG_LIB_PATH = os.path.join(PKG, "libattn_fwd_debug.so")

_lib = None


class AttnError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"{message} (status {code})")
        self.code = code


def header_functions() -> list[str]:
    """Names of the functions declared in include/attn_api.h."""
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(attn_\w+)\s*\(", text, flags=re.M)


def _declare(lib):
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, vp]
    lib.attn_fwd.restype = i
    lib.attn_fwd_padded.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, vp]
    lib.attn_fwd_padded.restype = i
    lib.attn_fwd_o32.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, vp]
    lib.attn_fwd_o32.restype = i
    lib.attn_fwd_decode_workspace_size.argtypes = [i, i, i, i, i, i, i]
    lib.attn_fwd_decode_workspace_size.restype = ctypes.c_size_t
    lib.attn_fwd_decode.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, i, vp,
                                    ctypes.c_size_t, vp]
    lib.attn_fwd_decode.restype = i
    lib.attn_fwd_decode_noalloc.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, i, f, i, vp]
    lib.attn_fwd_decode_noalloc.restype = i
    lib.attn_quantize_e4m3.argtypes = [vp, vp, vp, i, i, i, vp]
    lib.attn_quantize_e4m3_hadamard.argtypes = [vp, ctypes.c_uint64, ctypes.c_uint64, vp, vp, i, i, i, vp]
    lib.attn_quantize_e4m3_hadamard.restype = i
    lib.attn_quantize_e4m3.restype = i
    lib.attn_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, vp]
    lib.attn_fwd_fp8.restype = i
    lib.attn_fwd_host.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, vp]
    lib.attn_fwd_host.restype = i
    lib.attn_bwd_workspace_size.argtypes = [i, i, i, i]
    lib.attn_bwd_workspace_size.restype = ctypes.c_size_t
    lib.attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, vp, ctypes.c_size_t,
                             vp]
    lib.attn_bwd.restype = i
    lib.attn_status_str.argtypes = [i]
    lib.attn_status_str.restype = ctypes.c_char_p
    lib.attn_last_cuda_error.argtypes = []
    lib.attn_last_cuda_error.restype = i
    lib.attn_device_error.argtypes = [i]
    lib.attn_device_error.restype = i
    lib.attn_selftest_wait_timeout.argtypes = [ctypes.c_int64]
    lib.attn_selftest_wait_timeout.restype = i
    lib.attn_version.argtypes = []
    lib.attn_version.restype = i
    lib.attn_debug_build.argtypes = []
    lib.attn_debug_build.restype = i
    lib.attn_debug_first_site.argtypes = [i]
    lib.attn_debug_first_site.restype = i
    lib.attn_debug_selftest.argtypes = []
    lib.attn_debug_selftest.restype = i
    return lib


def load(path: str | None = None):
    """Load the CUDA library (built in-tree by exact_self_attention_fwd_b300.build)."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is missing: build it with `python -m exact_self_attention_fwd_b300.build`"
                " (there is no fallback implementation)")
        _lib = _declare(ctypes.CDLL(LIB_PATH))
    return _lib


@contextlib.contextmanager
def using(lib):
    """Route this module's wrappers through another build of the library (for
    example the debug build, load(DEBUG_LIB_PATH)) inside a `with` block."""
    global _lib
    old = _lib
    _lib = lib
    try:
        yield lib
    finally:
        _lib = old


def status_str(code: int) -> str:
    return load().attn_status_str(int(code)).decode()


def _check(rc: int):
    if rc != ATTN_OK:
        L = load()
        msg = L.attn_status_str(rc).decode()
        if rc == ATTN_ERR_CUDA:
            msg += f"; cudaError {L.attn_last_cuda_error()}"
        raise AttnError(rc, msg)


def _stream_handle(stream, device):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _check_tensors(q, k, v):
    import torch
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be 4-D [B, H, N, d]")
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.bfloat16:
            raise ValueError(f"{name} must be bfloat16")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    B, Hq, N, d = q.shape
    if k.shape != v.shape or k.shape[0] != B or k.shape[2] != N or k.shape[3] != d:
        raise ValueError("k and v must be [B, Hkv, N, d] matching q")
    return B, Hq, k.shape[1], N, d


def attn_fwd(q, k, v, causal: bool = False, window: int = 0, scale: float | None = None,
             out=None, lse=None, stream=None, key_len=None, out_fp32: bool = False):
    """O [B,Hq,N,d] bf16 and LSE [B,Hq,N] fp32 for CUDA bf16 q [B,Hq,N,d], k/v [B,Hkv,N,d].

    key_len: optional CUDA int32 [B] of valid lengths (right padding; attn_fwd_padded).
    out_fp32: write O as fp32 instead (attn_fwd_o32: the same kernel, O not rounded to
    bf16), to see the kernel's error apart from the output format.
    Asynchronous on `stream` (default: the current stream of q's device).
    """
    import torch
    B, Hq, Hkv, N, d = _check_tensors(q, k, v)
    dev = q.device
    if dev.type != "cuda" or k.device != dev or v.device != dev:
        raise ValueError("q, k, v must be CUDA tensors on one device")
    if scale is None:
        scale = d ** -0.5
    o_dtype = torch.float32 if out_fp32 else torch.bfloat16
    if out is None:
        out = torch.empty(q.shape, dtype=o_dtype, device=dev)
    if lse is None:
        lse = torch.empty((B, Hq, N), dtype=torch.float32, device=dev)
    if out.shape != q.shape or out.dtype != o_dtype or not out.is_contiguous() or out.device != dev:
        raise ValueError(f"out must be a contiguous {o_dtype} CUDA tensor shaped like q")
    if tuple(lse.shape) != (B, Hq, N) or lse.dtype != torch.float32 or not lse.is_contiguous() or lse.device != dev:
        raise ValueError("lse must be a contiguous fp32 CUDA tensor [B, Hq, N]")
    L = load()
    if key_len is not None:
        if (key_len.device != dev or key_len.dtype != torch.int32 or key_len.numel() != B
                or not key_len.is_contiguous()):
            raise ValueError("key_len must be a contiguous int32 CUDA tensor with B entries")
    with torch.cuda.device(dev):
        if out_fp32:
            rc = L.attn_fwd_o32(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                None if key_len is None else key_len.data_ptr(), B, Hq, Hkv, N, d,
                                int(bool(causal)), int(window), float(scale), _stream_handle(stream, dev))
        elif key_len is None:
            rc = L.attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                            B, Hq, Hkv, N, d, int(bool(causal)), int(window), float(scale),
                            _stream_handle(stream, dev))
        else:
            rc = L.attn_fwd_padded(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                   lse.data_ptr(), key_len.data_ptr(), B, Hq, Hkv, N, d,
                                   int(bool(causal)), int(window), float(scale),
                                   _stream_handle(stream, dev))
    _check(rc)
    return out, lse


def bwd_workspace_size(B: int, Hq: int, N: int, d: int) -> int:
    """Bytes of workspace attn_bwd needs (lse log2(e) and D = rowsum(dO o O) per query
    row, fp32, rows padded to a multiple of 128)."""
    return int(load().attn_bwd_workspace_size(B, Hq, N, d))


def bwd_row_sums(workspace, B: int, Hq: int, N: int):
    """View of D = rowsum(dO o O) that attn_bwd wrote into `workspace`: fp32 [B, Hq, N]
    (the workspace holds lse log2(e) and then D, each head's rows padded to a multiple
    of 128)."""
    import torch
    n_pad = (N + 127) // 128 * 128
    f = workspace[: 2 * B * Hq * n_pad * 4].view(torch.float32)
    return f[B * Hq * n_pad:].view(B, Hq, n_pad)[:, :, :N]


def attn_bwd(q, k, v, out, lse, dout, causal: bool = False, window: int = 0, scale: float | None = None,
             key_len=None, dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Gradients (dq [B,Hq,N,d], dk, dv [B,Hkv,N,d], all bf16) of attn_fwd's output for the
    upstream gradient dout [B,Hq,N,d] bf16; out and lse are the forward's results for the
    same q, k, v, mask and scale. workspace: a uint8 CUDA tensor of at least
    bwd_workspace_size(B, Hq, N, d) bytes (allocated when None). Asynchronous on `stream`.
    """
    import torch
    B, Hq, Hkv, N, d = _check_tensors(q, k, v)
    dev = q.device
    if dev.type != "cuda" or k.device != dev or v.device != dev:
        raise ValueError("q, k, v must be CUDA tensors on one device")
    for name, t in (("out", out), ("dout", dout)):
        if t.shape != q.shape or t.dtype != torch.bfloat16 or not t.is_contiguous() or t.device != dev:
            raise ValueError(f"{name} must be a contiguous bf16 CUDA tensor shaped like q")
    if tuple(lse.shape) != (B, Hq, N) or lse.dtype != torch.float32 or not lse.is_contiguous() or lse.device != dev:
        raise ValueError("lse must be a contiguous fp32 CUDA tensor [B, Hq, N]")
    if scale is None:
        scale = d ** -0.5
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for name, t, ref in (("dq", dq, q), ("dk", dk, k), ("dv", dv, v)):
        if t.shape != ref.shape or t.dtype != torch.bfloat16 or not t.is_contiguous() or t.device != dev:
            raise ValueError(f"{name} must be a contiguous bf16 CUDA tensor shaped like its input")
    need = bwd_workspace_size(B, Hq, N, d)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    if workspace.device != dev or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor on q's device")
    if key_len is not None and (key_len.device != dev or key_len.dtype != torch.int32 or key_len.numel() != B
                                or not key_len.is_contiguous()):
        raise ValueError("key_len must be a contiguous int32 CUDA tensor with B entries")
    L = load()
    with torch.cuda.device(dev):
        rc = L.attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                        dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                        None if key_len is None else key_len.data_ptr(), B, Hq, Hkv, N, d,
                        int(bool(causal)), int(window), float(scale), workspace.data_ptr(),
                        workspace.numel() * workspace.element_size(), _stream_handle(stream, dev))
    _check(rc)
    return dq, dk, dv


def decode_workspace_size(B: int, Hq: int, Hkv: int, Nq: int, Nk: int, d: int, splits: int = 0) -> int:
    """Bytes of workspace attn_fwd_decode needs (0 when it runs unsplit)."""
    return int(load().attn_fwd_decode_workspace_size(B, Hq, Hkv, Nq, Nk, d, int(splits)))


def attn_fwd_decode(q, k, v, causal: bool = True, window: int = 0, scale: float | None = None,
                    splits: int = 0, out=None, lse=None, workspace=None, stream=None):
    """Decode shape: CUDA bf16 q [B,Hq,Nq,d] are the last Nq positions of a sequence whose
    keys and values are k, v [B,Hkv,Nk,d]. Returns (o [B,Hq,Nq,d] bf16, lse [B,Hq,Nq] fp32).

    splits: parts of the key sequence computed by separate CTAs (0 = the library's
    choice). The fp32 workspace for the partial results is allocated here with torch
    when not given (uint8 CUDA tensor of at least decode_workspace_size(...) bytes)."""
    import torch
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be 4-D")
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.bfloat16 or not t.is_contiguous() or t.device.type != "cuda":
            raise ValueError(f"{name} must be a contiguous bf16 CUDA tensor")
    B, Hq, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    if k.shape != v.shape or k.shape[0] != B or k.shape[3] != d:
        raise ValueError("k and v must be [B, Hkv, Nk, d] matching q")
    dev = q.device
    if scale is None:
        scale = d ** -0.5
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=dev)
    L = load()
    with torch.cuda.device(dev):
        need = int(L.attn_fwd_decode_workspace_size(B, Hq, Hkv, Nq, Nk, d, int(splits)))
        if workspace is None and need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=dev)
        ws_ptr = workspace.data_ptr() if workspace is not None else None
        ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
        rc = L.attn_fwd_decode(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                               B, Hq, Hkv, Nq, Nk, d, int(bool(causal)), int(window), float(scale),
                               int(splits), ws_ptr, ws_bytes, _stream_handle(stream, dev))
    _check(rc)
    return out, lse


def quantize_e4m3(x, stream=None):
    """Block quantisation of a CUDA bf16 tensor [..., N, d] (d = 64 or 128) to e4m3 codes
    (uint8, same shape) and fp32 scales [heads, ceil(N / 128)] (attn_quantize_e4m3)."""
    import torch
    if x.dtype != torch.bfloat16 or not x.is_contiguous() or x.device.type != "cuda" or x.dim() < 2:
        raise ValueError("x must be a contiguous bf16 CUDA tensor [..., N, d]")
    N, d = x.shape[-2], x.shape[-1]
    BH = x.numel() // (N * d)
    codes = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    scales = torch.empty((BH, (N + 127) // 128), dtype=torch.float32, device=x.device)
    with torch.cuda.device(x.device):
        rc = load().attn_quantize_e4m3(x.data_ptr(), codes.data_ptr(), scales.data_ptr(), BH, N, d,
                                       _stream_handle(stream, x.device))
    _check(rc)
    return codes, scales


def sign_masks(signs) -> tuple[int, int]:
    """The two 64-bit masks of attn_quantize_e4m3_hadamard for 128 signs (+1 or -1):
    bit c set where signs[c] is -1."""
    sg = [float(x) for x in signs]
    if len(sg) != 128 or any(x not in (1.0, -1.0) for x in sg):
        raise ValueError("signs must be 128 values, each +1 or -1")
    bits = sum(1 << c for c, x in enumerate(sg) if x < 0)
    return bits & ((1 << 64) - 1), bits >> 64


def quantize_e4m3_hadamard(x, signs, stream=None):
    """Incoherent processing (x M, M = diag(signs) H / sqrt(128)) then block quantisation
    of a CUDA bf16 tensor [..., N, 128]: e4m3 codes (uint8, same shape) and fp32 scales
    [heads, ceil(N / 128)] (attn_quantize_e4m3_hadamard). Use the same signs for Q and K."""
    import torch
    if x.dtype != torch.bfloat16 or not x.is_contiguous() or x.device.type != "cuda" or x.dim() < 2:
        raise ValueError("x must be a contiguous bf16 CUDA tensor [..., N, d]")
    N, d = x.shape[-2], x.shape[-1]
    BH = x.numel() // (N * d)
    lo, hi = sign_masks(signs)
    codes = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    scales = torch.empty((BH, (N + 127) // 128), dtype=torch.float32, device=x.device)
    with torch.cuda.device(x.device):
        rc = load().attn_quantize_e4m3_hadamard(x.data_ptr(), lo, hi, codes.data_ptr(), scales.data_ptr(), BH, N,
                                                d, _stream_handle(stream, x.device))
    _check(rc)
    return codes, scales


def attn_fwd_fp8(q8, k8, v8, q_scale, k_scale, v_scale, causal: bool = False, window: int = 0,
                 scale: float | None = None, out=None, lse=None, stream=None):
    """Attention forward on e4m3 operands with per-block scales (attn_fwd_fp8): q8
    [B,Hq,N,128], k8/v8 [B,Hkv,N,128] uint8 codes, scales fp32 [B*H, ceil(N/128)] as
    quantize_e4m3 makes them. Returns (o bf16 [B,Hq,N,128], lse fp32 [B,Hq,N])."""
    import torch
    for name, t in (("q8", q8), ("k8", k8), ("v8", v8)):
        if t.dtype != torch.uint8 or not t.is_contiguous() or t.device.type != "cuda" or t.dim() != 4:
            raise ValueError(f"{name} must be a contiguous 4-D uint8 CUDA tensor")
    for name, t in (("q_scale", q_scale), ("k_scale", k_scale), ("v_scale", v_scale)):
        if t.dtype != torch.float32 or not t.is_contiguous() or t.device.type != "cuda":
            raise ValueError(f"{name} must be a contiguous fp32 CUDA tensor")
    B, Hq, N, d = q8.shape
    Hkv = k8.shape[1]
    if k8.shape != v8.shape or k8.shape[0] != B or k8.shape[2] != N or k8.shape[3] != d:
        raise ValueError("k8 and v8 must be [B, Hkv, N, d] matching q8")
    nblk = (N + 127) // 128
    if q_scale.numel() != B * Hq * nblk or k_scale.numel() != B * Hkv * nblk or v_scale.numel() != B * Hkv * nblk:
        raise ValueError("scales must have one entry per 128-row block of every head")
    dev = q8.device
    if scale is None:
        scale = d ** -0.5
    if out is None:
        out = torch.empty((B, Hq, N, d), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((B, Hq, N), dtype=torch.float32, device=dev)
    with torch.cuda.device(dev):
        rc = load().attn_fwd_fp8(q8.data_ptr(), k8.data_ptr(), v8.data_ptr(), q_scale.data_ptr(),
                                 k_scale.data_ptr(), v_scale.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                 B, Hq, Hkv, N, d, int(bool(causal)), int(window), float(scale),
                                 _stream_handle(stream, dev))
    _check(rc)
    return out, lse


def attn_fwd_host(hq, hk, hv, ho, hlse, dq, dk, dv, do, dlse, causal: bool = False,
                  window: int = 0, scale: float | None = None, stream=None):
    """Host-buffer entry: copies hq/hk/hv into dq/dk/dv, runs, copies do/dlse back into
    ho/hlse, pipelined over chunks of (batch, KV head) groups so that copies overlap the
    kernels (the copies run on two library-owned streams, ordered against `stream`).
    Host tensors should be pinned; synchronise `stream` before reading ho and hlse."""
    import torch
    B, Hq, Hkv, N, d = _check_tensors(hq, hk, hv)
    _check_tensors(dq, dk, dv)
    dev = dq.device
    if scale is None:
        scale = d ** -0.5
    for t in (hq, hk, hv, ho, hlse):
        if t.device.type != "cpu":
            raise ValueError("host buffers must be CPU tensors")
    for t in (dq, dk, dv, do, dlse):
        if t.device != dev or dev.type != "cuda":
            raise ValueError("device buffers must be CUDA tensors on one device")
    if ho.shape != hq.shape or do.shape != hq.shape or dq.shape != hq.shape or dk.shape != hk.shape:
        raise ValueError("buffer shapes do not match")
    if tuple(hlse.shape) != (B, Hq, N) or tuple(dlse.shape) != (B, Hq, N):
        raise ValueError("lse buffers must be [B, Hq, N]")
    L = load()
    with torch.cuda.device(dev):
        rc = L.attn_fwd_host(hq.data_ptr(), hk.data_ptr(), hv.data_ptr(), ho.data_ptr(), hlse.data_ptr(),
                             dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), do.data_ptr(), dlse.data_ptr(),
                             B, Hq, Hkv, N, d, int(bool(causal)), int(window), float(scale),
                             _stream_handle(stream, dev))
    _check(rc)
    return ho, hlse


def device_error(clear: bool = True) -> int:
    """Synchronise and return ATTN_OK or ATTN_ERR_TIMEOUT (see attn_device_error)."""
    return load().attn_device_error(int(bool(clear)))


def selftest_wait_timeout(limit_ns: int) -> int:
    return load().attn_selftest_wait_timeout(int(limit_ns))


def version() -> int:
    return load().attn_version()
