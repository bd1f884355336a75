"""Failure detection without a GPU fault: a bounded pipeline wait that nothing
completes runs out, the kernel records ATTN_ERR_TIMEOUT in the device status word
and returns, and the context stays usable for the next call."""
import math

import pytest
import torch

import oracle
import exact_self_attention_fwd_b300 as ea
from exact_self_attention_fwd_b300.inputs import make_qkv
from parity import compare

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_context_survives():
    assert ea.device_error(clear=True) == ea.ATTN_OK
    assert ea.selftest_wait_timeout(20_000_000) == ea.ATTN_ERR_TIMEOUT  # 20 ms
    # the status word was cleared by the self-test; a normal call works afterwards
    assert ea.device_error(clear=True) == ea.ATTN_OK
    q, k, v = make_qkv(1, 2, 2, 200, 64, 21)
    out, lse = ea.attn_fwd(q.cuda(), k.cuda(), v.cuda(), causal=True)
    torch.cuda.synchronize()
    assert ea.device_error() == ea.ATTN_OK
    o_ref, l_ref = oracle.attn_ref(q, k, v, causal=True, scale=1 / math.sqrt(64))
    compare(out, lse, o_ref, l_ref, "after timeout self-test")
