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
