"""fp64 CPU oracle for exact scaled-dot-product attention forward.

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` are the only permitted users. The
product library never imports, links or calls anything here, and this package
imports nothing from the product package.

The arithmetic lives in ``attn_ref.c`` (plain C, fp64, one thread per slice of
rows); this module only compiles it with gcc and marshals numpy arrays.

Parity status of each function (see the pins in ``tests/test_oracle_pins.py`` and
``tests/test_oracle_fp8.py``):
  attn_ref / attn_ref_rows -- pinned (closed forms, invariants, brute force,
  an independent library routine, and mutation tests).
  attn_ref_decode -- pinned (the last rows of the plain forward, a zero-query closed
  form, brute force and torch SDPA with an offset mask).
  attn_ref_bwd -- pinned (torch autograd through fp64 scaled_dot_product_attention with
  the same masks, central finite differences of the oracle's own forward, and the
  invariants sum_j ds_ij = 0 and dv = sum of p^T do). Its given-o form is pinned by
  equality with the chain-rule form for the exact o and by the closed-form response to
  a change of one element of o; attn_ref_bwd_dq_rows by equality with its dq on every
  row.
  e4m3_encode / e4m3_decode / quantize_e4m3_blocks / attn_ref_fp8 -- pinned (every code
  against torch's float8_e4m3fn, the rounding of every bf16 value in range, block
  reconstruction bounds, exactness on representable inputs, and the block-vs-tensor
  scaling error comparison the FlashAttention-3 review reports).
  hadamard / incoherent / quantize_e4m3_blocks_f64 / attn_ref_fp8(signs=...) -- pinned
  (the Sylvester matrix against scipy's and H H^T = d I, one-hot rows, preserved scores
  and attention, quantiser bounds and agreement with the fp32 quantiser where both scale
  by exactly 1, and lower error with outlier channels).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_ref.c")
_LIB = os.path.join(_HERE, "libattn_ref.so")

_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile the oracle with gcc (strict IEEE fp64: no fast-math)."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    tmp = out + ".tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
           "-fno-fast-math", "-ffp-contract=off", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _declare(lib):
    u16p = ctypes.POINTER(ctypes.c_uint16)
    f64p = ctypes.POINTER(ctypes.c_double)
    i64p = ctypes.POINTER(ctypes.c_int64)
    i64 = ctypes.c_int64
    i32p = ctypes.POINTER(ctypes.c_int32)
    lib.attn_ref_fwd_rows_f64.argtypes = [
        u16p, u16p, u16p, i64, i64, i64, i64, i64, ctypes.c_int, i64, ctypes.c_double,
        i32p, i64p, i64, f64p, f64p, ctypes.c_int]
    lib.attn_ref_fwd_rows_f64.restype = ctypes.c_int
    lib.attn_ref_fwd_f64.argtypes = [
        u16p, u16p, u16p, i64, i64, i64, i64, i64, ctypes.c_int, i64, ctypes.c_double,
        i32p, f64p, f64p, ctypes.c_int]
    lib.attn_ref_fwd_f64.restype = ctypes.c_int
    lib.attn_ref_decode_rows_f64.argtypes = [
        u16p, u16p, u16p, i64, i64, i64, i64, i64, i64, ctypes.c_int, i64, ctypes.c_double,
        i64p, i64, f64p, f64p, ctypes.c_int]
    lib.attn_ref_decode_rows_f64.restype = ctypes.c_int
    lib.attn_ref_fwd_rows_f64in.argtypes = [
        f64p, f64p, f64p, i64, i64, i64, i64, i64, ctypes.c_int, i64, ctypes.c_double,
        i64p, i64, f64p, f64p, ctypes.c_int]
    lib.attn_ref_fwd_rows_f64in.restype = ctypes.c_int
    u8p = ctypes.POINTER(ctypes.c_uint8)
    lib.attn_ref_e4m3_decode.argtypes = [u8p, i64, f64p]
    lib.attn_ref_e4m3_decode.restype = None
    lib.attn_ref_e4m3_encode.argtypes = [f64p, i64, u8p]
    lib.attn_ref_e4m3_encode.restype = None
    lib.attn_ref_quantize_e4m3_blocks.argtypes = [u16p, i64, i64, i64, i64, u8p,
                                                  ctypes.POINTER(ctypes.c_float)]
    lib.attn_ref_quantize_e4m3_blocks.restype = ctypes.c_int
    lib.attn_ref_bwd_f64.argtypes = [u16p, u16p, u16p, u16p, i64, i64, i64, i64, i64, ctypes.c_int, i64,
                                     ctypes.c_double, ctypes.POINTER(ctypes.c_int32), f64p, f64p, f64p,
                                     ctypes.c_int]
    lib.attn_ref_bwd_f64.restype = ctypes.c_int
    lib.attn_ref_bwd_dq_rows_f64.argtypes = [u16p, u16p, u16p, u16p, i64, i64, i64, i64, i64, ctypes.c_int, i64,
                                             ctypes.c_double, ctypes.POINTER(ctypes.c_int32),
                                             ctypes.POINTER(ctypes.c_int64), i64, f64p]
    lib.attn_ref_bwd_dq_rows_f64.restype = ctypes.c_int
    lib.attn_ref_quantize_e4m3_blocks_f64.argtypes = [f64p, i64, i64, i64, i64, ctypes.POINTER(ctypes.c_uint8),
                                                      f64p]
    lib.attn_ref_quantize_e4m3_blocks_f64.restype = ctypes.c_int
    lib.attn_ref_bwd_given_o_f64.argtypes = [u16p, u16p, u16p, u16p, f64p, i64, i64, i64, i64, i64, ctypes.c_int,
                                             i64, ctypes.c_double, ctypes.POINTER(ctypes.c_int32), f64p, f64p,
                                             f64p, ctypes.c_int]
    lib.attn_ref_bwd_given_o_f64.restype = ctypes.c_int
    return lib


def load(path: str | None = None):
    """Load (building first if needed) the oracle shared library."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    if _lib is None:
        build()
        _lib = _declare(ctypes.CDLL(_LIB))
    return _lib


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def _as_bits(x) -> np.ndarray:
    """Accept uint16 bf16 bit patterns (numpy) or a torch bfloat16 tensor."""
    if isinstance(x, np.ndarray):
        if x.dtype != np.uint16:
            raise TypeError("oracle inputs are bf16 bit patterns (numpy uint16)")
        return np.ascontiguousarray(x)
    # torch tensor (CPU, bfloat16): reinterpret the bits without arithmetic
    import torch
    if x.dtype != torch.bfloat16:
        raise TypeError("oracle inputs must be bfloat16")
    return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def attn_ref_rows(q, k, v, causal: bool, window: int, scale: float, rows=None,
                  nthreads: int | None = None, lib=None, key_len=None):
    """fp64 O and LSE for the listed flat rows ((b*Hq)+hq)*N + i (all rows if None).

    q: [B,Hq,N,d], k/v: [B,Hkv,N,d] bf16; key_len: optional per-batch valid length
    (right padding). Returns (o [nrows,d] f64, lse [nrows] f64); a row with no visible
    key has o = 0 and lse = -inf.
    """
    qb, kb, vb = _as_bits(q), _as_bits(k), _as_bits(v)
    B, Hq, N, d = qb.shape
    Hkv = kb.shape[1]
    if kb.shape != (B, Hkv, N, d) or vb.shape != kb.shape:
        raise ValueError("k and v must be [B,Hkv,N,d] matching q")
    if rows is None:
        nrows = B * Hq * N
        rows_arr = None
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        nrows = rows_arr.size
    kl = None
    if key_len is not None:
        kl = np.ascontiguousarray(np.asarray(key_len, dtype=np.int32).reshape(-1))
        if kl.size != B:
            raise ValueError("key_len must have one entry per batch")
    o = np.empty((nrows, d), dtype=np.float64)
    lse = np.empty((nrows,), dtype=np.float64)
    L = lib or load()
    u16p = ctypes.POINTER(ctypes.c_uint16)
    f64p = ctypes.POINTER(ctypes.c_double)
    rc = L.attn_ref_fwd_rows_f64(
        qb.ctypes.data_as(u16p), kb.ctypes.data_as(u16p), vb.ctypes.data_as(u16p),
        B, Hq, Hkv, N, d, int(bool(causal)), int(window), float(scale),
        kl.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)) if kl is not None else None,
        rows_arr.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)) if rows_arr is not None else None,
        nrows, o.ctypes.data_as(f64p), lse.ctypes.data_as(f64p),
        int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (code {rc})")
    return o, lse


def attn_ref(q, k, v, causal: bool = False, window: int = 0, scale: float | None = None,
             nthreads: int | None = None, lib=None, key_len=None):
    """fp64 O [B,Hq,N,d] and LSE [B,Hq,N] for every row."""
    qb = _as_bits(q)
    B, Hq, N, d = qb.shape
    if scale is None:
        scale = 1.0 / float(np.sqrt(d))
    o, lse = attn_ref_rows(qb, k, v, causal, window, scale, None, nthreads, lib, key_len)
    return o.reshape(B, Hq, N, d), lse.reshape(B, Hq, N)


def attn_ref_decode(q, k, v, causal: bool = True, window: int = 0, scale: float | None = None,
                    rows=None, nthreads: int | None = None, lib=None):
    """Decode shape: q [B,Hq,Nq,d] are the last Nq positions of a sequence whose keys
    and values k, v are [B,Hkv,Nk,d]. Returns fp64 (o, lse) shaped [B,Hq,Nq,d] and
    [B,Hq,Nq], or [nrows,d] and [nrows] for a list of flat rows ((b*Hq)+hq)*Nq + i."""
    qb, kb, vb = _as_bits(q), _as_bits(k), _as_bits(v)
    B, Hq, Nq, d = qb.shape
    Hkv, Nk = kb.shape[1], kb.shape[2]
    if kb.shape != (B, Hkv, Nk, d) or vb.shape != kb.shape:
        raise ValueError("k and v must be [B,Hkv,Nk,d] matching q")
    if scale is None:
        scale = 1.0 / float(np.sqrt(d))
    rows_arr = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    nrows = B * Hq * Nq if rows_arr is None else rows_arr.size
    o = np.empty((nrows, d), dtype=np.float64)
    lse = np.empty((nrows,), dtype=np.float64)
    L = lib or load()
    u16p = ctypes.POINTER(ctypes.c_uint16)
    f64p = ctypes.POINTER(ctypes.c_double)
    rc = L.attn_ref_decode_rows_f64(
        qb.ctypes.data_as(u16p), kb.ctypes.data_as(u16p), vb.ctypes.data_as(u16p),
        B, Hq, Hkv, Nq, Nk, d, int(bool(causal)), int(window), float(scale),
        rows_arr.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)) if rows_arr is not None else None,
        nrows, o.ctypes.data_as(f64p), lse.ctypes.data_as(f64p), int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (code {rc})")
    if rows_arr is None:
        return o.reshape(B, Hq, Nq, d), lse.reshape(B, Hq, Nq)
    return o, lse


# ---------------------------------------------------------------- FP8 (e4m3) blocks
def e4m3_decode(codes) -> np.ndarray:
    """fp64 values of e4m3 codes (uint8 array)."""
    c = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8))
    out = np.empty(c.shape, dtype=np.float64)
    load().attn_ref_e4m3_decode(c.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)), c.size,
                                out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    return out


def e4m3_encode(x) -> np.ndarray:
    """Nearest e4m3 code (ties to even, saturating at 448) of each finite fp64 value."""
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    out = np.empty(a.shape, dtype=np.uint8)
    load().attn_ref_e4m3_encode(a.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), a.size,
                                out.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)))
    return out


def quantize_e4m3_blocks(x, rows: int = 128):
    """Block quantisation of bf16 x [..., N, d] (leading dims flattened to heads): codes
    (uint8, same shape) and scales (fp32 [heads, ceil(N / rows)])."""
    xb = _as_bits(x)
    *lead, N, d = xb.shape
    BH = int(np.prod(lead)) if lead else 1
    codes = np.empty(xb.shape, dtype=np.uint8)
    nblk = (N + rows - 1) // rows
    scales = np.empty((BH, nblk), dtype=np.float32)
    rc = load().attn_ref_quantize_e4m3_blocks(
        xb.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16)), BH, N, d, rows,
        codes.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)),
        scales.ctypes.data_as(ctypes.POINTER(ctypes.c_float)))
    if rc != 0:
        raise ValueError("bad arguments")
    return codes, scales


def dequantize_e4m3_blocks(codes, scales, rows: int = 128) -> np.ndarray:
    """fp64 code x scale of each element."""
    c = np.asarray(codes)
    *lead, N, d = c.shape
    BH = int(np.prod(lead)) if lead else 1
    vals = e4m3_decode(c).reshape(BH, N, d)
    sc = np.asarray(scales, dtype=np.float64).reshape(BH, -1)
    blk = np.arange(N) // rows
    return (vals * sc[:, blk][:, :, None]).reshape(c.shape)


def attn_ref_f64in(q, k, v, causal: bool = False, window: int = 0, scale: float = 1.0,
                   rows=None, nthreads: int | None = None):
    """The plain forward on fp64 inputs q [B,Hq,N,d], k/v [B,Hkv,N,d]."""
    qa, ka, va = (np.ascontiguousarray(np.asarray(t, dtype=np.float64)) for t in (q, k, v))
    B, Hq, N, d = qa.shape
    Hkv = ka.shape[1]
    rows_arr = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    nrows = B * Hq * N if rows_arr is None else rows_arr.size
    o = np.empty((nrows, d), dtype=np.float64)
    lse = np.empty((nrows,), dtype=np.float64)
    f64p = ctypes.POINTER(ctypes.c_double)
    rc = load().attn_ref_fwd_rows_f64in(
        qa.ctypes.data_as(f64p), ka.ctypes.data_as(f64p), va.ctypes.data_as(f64p), B, Hq, Hkv, N, d,
        int(bool(causal)), int(window), float(scale),
        rows_arr.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)) if rows_arr is not None else None,
        nrows, o.ctypes.data_as(f64p), lse.ctypes.data_as(f64p), int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (code {rc})")
    if rows_arr is None:
        return o.reshape(B, Hq, N, d), lse.reshape(B, Hq, N)
    return o, lse


def attn_ref_bwd_dq_rows(q, k, v, do, rows, causal: bool = False, window: int = 0,
                         scale: float | None = None, key_len=None, lib=None):
    """fp64 query gradients [len(rows), d] of the flat query rows (b * Hq + hq) * N + i,
    each computed from its own row (the exact row term D), for full-size checks."""
    qb, kb, vb, db = (_as_bits(t) for t in (q, k, v, do))
    B, Hq, N, d = qb.shape
    Hkv = kb.shape[1]
    if scale is None:
        scale = 1.0 / float(np.sqrt(d))
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    out = np.empty((len(r), d), dtype=np.float64)
    kl = None if key_len is None else np.ascontiguousarray(np.asarray(key_len, dtype=np.int32))
    u16p = ctypes.POINTER(ctypes.c_uint16)
    rc = (lib or load()).attn_ref_bwd_dq_rows_f64(
        qb.ctypes.data_as(u16p), kb.ctypes.data_as(u16p), vb.ctypes.data_as(u16p), db.ctypes.data_as(u16p),
        B, Hq, Hkv, N, d, int(bool(causal)), int(window), float(scale),
        kl.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)) if kl is not None else None,
        r.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), len(r),
        out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (code {rc})")
    return out


def hadamard(d: int) -> np.ndarray:
    """The Sylvester Hadamard matrix of order d (a power of two), entries +-1, fp64:
    H_1 = [1], H_2n = [[H_n, H_n], [H_n, -H_n]], so H H^T = d I."""
    if d < 1 or d & (d - 1):
        raise ValueError("d must be a power of two")
    h = np.ones((1, 1))
    while h.shape[0] < d:
        h = np.block([[h, h], [h, -h]])
    return h


def incoherent(x, signs) -> np.ndarray:
    """Incoherent processing of the FlashAttention-3 review: x' = x M with the random
    orthogonal M = diag(signs) H / sqrt(d) (signs +-1, H the Sylvester Hadamard
    matrix). x bf16 (or real) [..., d]; returns fp64 [..., d]. Since M M^T = I,
    Q' K'^T = Q K^T: attention on (Q', K', V) is attention on (Q, K, V)."""
    xv = x.double().numpy() if hasattr(x, "double") else np.asarray(x, dtype=np.float64)
    s = np.asarray(signs, dtype=np.float64)
    d = xv.shape[-1]
    return (xv * s) @ hadamard(d) / np.sqrt(d)


def quantize_e4m3_blocks_f64(x, rows: int = 128):
    """Block quantisation of real values x [..., N, d] (fp64, exact arithmetic): codes
    uint8 [..., N, d] and fp64 scales [heads, ceil(N / rows)] with scale = amax / 448."""
    xv = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    *lead, N, d = xv.shape
    BH = int(np.prod(lead)) if lead else 1
    codes = np.empty(xv.shape, dtype=np.uint8)
    nblk = (N + rows - 1) // rows
    scales = np.empty((BH, nblk), dtype=np.float64)
    rc = load().attn_ref_quantize_e4m3_blocks_f64(
        xv.ctypes.data_as(ctypes.POINTER(ctypes.c_double)), BH, N, d, rows,
        codes.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)),
        scales.ctypes.data_as(ctypes.POINTER(ctypes.c_double)))
    if rc != 0:
        raise ValueError("bad arguments")
    return codes, scales


def attn_ref_fp8(q, k, v, causal: bool = False, window: int = 0, scale: float | None = None,
                 rows=None, block_rows: int = 128, per_tensor: bool = False, signs=None):
    """FP8 attention as the FlashAttention-3 review describes it: Q, K and V are block
    quantised to e4m3 (blocks of block_rows x d per head, or one scale for the whole
    tensor when per_tensor), then attention is computed exactly (fp64) on the
    dequantised values. With `signs` (+-1 per channel), Q and K first go through
    incoherent processing (x M, M = diag(signs) H / sqrt(d)) and their rotated values
    are block quantised in exact arithmetic. Returns (o, lse) like attn_ref, plus the
    dequantised inputs."""
    d = q.shape[-1]
    if scale is None:
        scale = 1.0 / float(np.sqrt(d))
    deq = []
    for i, t in enumerate((q, k, v)):
        if signs is not None and i < 2:
            codes, sc = quantize_e4m3_blocks_f64(incoherent(t, signs), rows=block_rows)
            deq.append(dequantize_e4m3_blocks(codes, sc, rows=block_rows))
        elif per_tensor:
            flat = t.reshape(1, 1, -1, d)
            codes, sc = quantize_e4m3_blocks(flat, rows=flat.shape[2])
            deq.append(dequantize_e4m3_blocks(codes, sc, rows=flat.shape[2]).reshape(tuple(t.shape)))
        else:
            codes, sc = quantize_e4m3_blocks(t, rows=block_rows)
            deq.append(dequantize_e4m3_blocks(codes, sc, rows=block_rows))
    o, lse = attn_ref_f64in(deq[0], deq[1], deq[2], causal, window, scale, rows)
    return o, lse, deq


def attn_ref_bwd(q, k, v, do, causal: bool = False, window: int = 0, scale: float | None = None,
                 key_len=None, lib=None, o=None, nthreads: int | None = None):
    """fp64 gradients (dq [B,Hq,N,d], dk, dv [B,Hkv,N,d]) of the forward's o for the
    upstream gradient do [B,Hq,N,d] (all inputs bf16).

    nthreads: threads over slices of query rows (default: every core this process may
    use); the dk, dv partials of the slices are added in slice order.

    o: None, or a given forward output [B,Hq,N,d] (any float type, taken as fp64): the
    softmax row sum of dp is then formed as do_i . o_i from it, as a backward pass that
    takes the forward's output as an input does (identical for the exact output)."""
    qb, kb, vb, db = (_as_bits(t) for t in (q, k, v, do))
    B, Hq, N, d = qb.shape
    Hkv = kb.shape[1]
    if scale is None:
        scale = 1.0 / float(np.sqrt(d))
    dq = np.empty((B, Hq, N, d), dtype=np.float64)
    dk = np.empty((B, Hkv, N, d), dtype=np.float64)
    dv = np.empty((B, Hkv, N, d), dtype=np.float64)
    kl = None if key_len is None else np.ascontiguousarray(np.asarray(key_len, dtype=np.int32))
    u16p = ctypes.POINTER(ctypes.c_uint16)
    f64p = ctypes.POINTER(ctypes.c_double)
    L = lib or load()
    if o is not None:
        ob = np.ascontiguousarray(np.asarray(o.double().numpy() if hasattr(o, "double") else o,
                                             dtype=np.float64).reshape(B, Hq, N, d))
        rc = L.attn_ref_bwd_given_o_f64(
            qb.ctypes.data_as(u16p), kb.ctypes.data_as(u16p), vb.ctypes.data_as(u16p), db.ctypes.data_as(u16p),
            ob.ctypes.data_as(f64p), B, Hq, Hkv, N, d, int(bool(causal)), int(window), float(scale),
            kl.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)) if kl is not None else None,
            dq.ctypes.data_as(f64p), dk.ctypes.data_as(f64p), dv.ctypes.data_as(f64p),
            int(nthreads or default_threads()))
        if rc != 0:
            raise ValueError(f"oracle rejected the arguments (code {rc})")
        return dq, dk, dv
    rc = L.attn_ref_bwd_f64(
        qb.ctypes.data_as(u16p), kb.ctypes.data_as(u16p), vb.ctypes.data_as(u16p), db.ctypes.data_as(u16p),
        B, Hq, Hkv, N, d, int(bool(causal)), int(window), float(scale),
        kl.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)) if kl is not None else None,
        dq.ctypes.data_as(f64p), dk.ctypes.data_as(f64p), dv.ctypes.data_as(f64p),
        int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (code {rc})")
    return dq, dk, dv
