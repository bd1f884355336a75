"""attn_fwd_decode_noalloc: the decode entry point that allocates nothing.

It is meant for callers that cannot allocate device memory while they run: a serving
loop whose memory budget was fixed at start-up, code running inside an allocator or
memory-pool callback (where the allocator must not be re-entered), or a plain C host
that holds only the tensors it passes. It keeps the split results in the library's
fixed scratch array instead of a caller workspace.

Each of two calls in a row (two shapes, both using the scratch) is checked against
attn_fwd_decode, the entry point that takes a workspace, within the parity tolerance
of the other tests. The file name makes pytest collect it last, so a run that stops
at the first failure has already run everything else; it also passes on its own in a
fresh process.
"""
import ctypes
import math

import pytest
import torch

import exact_self_attention_fwd_b300 as ea
from exact_self_attention_fwd_b300.inputs import make_qkv_decode
from parity import compare

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def call_noalloc(q, k, v, causal, window, scale, splits):
    """Through the C ABI: the caller passes only inputs and outputs."""
    B, Hq, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    o = torch.empty_like(q)
    lse = torch.empty((B, Hq, Nq), dtype=torch.float32, device=q.device)
    rc = ea.load().attn_fwd_decode_noalloc(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, Hq, Hkv, Nq, Nk, d,
        int(causal), int(window), float(scale), int(splits),
        ctypes.c_void_p(torch.cuda.current_stream(q.device).cuda_stream))
    return rc, o, lse


def test_noalloc_matches_workspace_entry_on_two_calls():
    cases = [
        # B, Hq, Hkv, Nq, Nk, d, causal, window, splits (0 = library's choice), seed
        (4, 32, 8, 1, 8192, 128, True, 0, 0, 11),
        (2, 16, 2, 4, 3000, 64, True, 500, 7, 12),
    ]
    for B, Hq, Hkv, Nq, Nk, d, causal, window, splits, seed in cases:
        q, k, v = make_qkv_decode(B, Hq, Hkv, Nq, Nk, d, seed)
        q, k, v = q.to(DEV), k.to(DEV), v.to(DEV)
        scale = 1.0 / math.sqrt(d)
        rc, o, lse = call_noalloc(q, k, v, causal, window, scale, splits)
        assert rc == ea.ATTN_OK, ea.status_str(rc)
        o_ref, lse_ref = ea.attn_fwd_decode(q, k, v, causal=causal, window=window, scale=scale,
                                            splits=splits)
        torch.cuda.synchronize()
        assert ea.device_error() == ea.ATTN_OK
        compare(o, lse, o_ref.double().cpu().numpy(), lse_ref.double().cpu().numpy(),
                f"no-alloc vs workspace B{B} Hq{Hq} Nq{Nq} Nk{Nk} d{d} splits {splits}")


def test_noalloc_rejects_results_beyond_its_scratch():
    # 16 x 64 heads x 16 queries, d = 128, two splits: about 17 MB of split results,
    # more than the fixed 8 MiB scratch holds
    q = torch.zeros(16, 64, 16, 128, dtype=torch.bfloat16, device=DEV)
    k = torch.zeros(16, 8, 256, 128, dtype=torch.bfloat16, device=DEV)
    rc, _, _ = call_noalloc(q, k, k, True, 0, 0.1, 2)
    assert rc == ea.ATTN_ERR_SCRATCH_LIMIT


LIMIT = 8 << 20  # ATTN_DECODE_NOALLOC_SCRATCH_BYTES


def test_noalloc_scratch_limit_boundary():
    # The split results of splits x B x Hq x Nq rows take rows x (4 d + 4) bytes at d = 64
    # (the 4 d part is already a multiple of the 256-byte alignment): 32263 rows
    # (7 splits x 419 x 11 heads x 1 query) are the most that fit in 8 MiB, 228 bytes
    # short of it; 32264 rows (8 x 109 x 37 x 1) are 32 bytes over.
    fit = (419, 11, 1, 1, 7 * 128, 64, 7)
    over = (109, 37, 1, 1, 8 * 128, 64, 8)
    B, Hq, Hkv, Nq, Nk, d, splits = fit
    assert ea.decode_workspace_size(B, Hq, Hkv, Nq, Nk, d, splits) == 32263 * 260 <= LIMIT
    q, k, v = make_qkv_decode(B, Hq, Hkv, Nq, Nk, d, 13)
    q, k, v = q.to(DEV), k.to(DEV), v.to(DEV)
    rc, o, lse = call_noalloc(q, k, v, True, 0, 0.125, splits)
    assert rc == ea.ATTN_OK, ea.status_str(rc)
    o_ref, lse_ref = ea.attn_fwd_decode(q, k, v, causal=True, scale=0.125, splits=splits)
    torch.cuda.synchronize()
    assert ea.device_error() == ea.ATTN_OK
    compare(o, lse, o_ref.double().cpu().numpy(), lse_ref.double().cpu().numpy(), "no-alloc at the limit")
    B, Hq, Hkv, Nq, Nk, d, splits = over
    assert ea.decode_workspace_size(B, Hq, Hkv, Nq, Nk, d, splits) == 32264 * 260 > LIMIT
    q = torch.zeros(B, Hq, Nq, d, dtype=torch.bfloat16, device=DEV)
    k = torch.zeros(B, Hkv, Nk, d, dtype=torch.bfloat16, device=DEV)
    rc, _, _ = call_noalloc(q, k, k, True, 0, 0.125, splits)
    assert rc == ea.ATTN_ERR_SCRATCH_LIMIT


def test_noalloc_rejects_the_librarys_own_split_count_beyond_its_scratch():
    # splits = 0: one KV head of 128 packed query rows against 1024 key tiles; the
    # library splits the keys over about one CTA per SM, and the split results of
    # that count do not fit
    B, Hq, Hkv, Nq, Nk, d = 1, 128, 1, 1, 1024 * 128, 128
    need = ea.decode_workspace_size(B, Hq, Hkv, Nq, Nk, d, 0)
    assert need > LIMIT
    q = torch.zeros(B, Hq, Nq, d, dtype=torch.bfloat16, device=DEV)
    k = torch.zeros(B, Hkv, Nk, d, dtype=torch.bfloat16, device=DEV)
    rc, _, _ = call_noalloc(q, k, k, True, 0, 0.1, 0)
    assert rc == ea.ATTN_ERR_SCRATCH_LIMIT
