"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module draws random numbers and nothing else: it holds none of the attention
arithmetic, so both the CUDA path and the CPU oracle can be fed from it without
sharing any of the method's code.

Recipe (one generator per workload):
  g = torch.Generator().manual_seed(seed)
  q = randn([B,Hq,N,d], fp32), then k = randn([B,Hkv,N,d]), then v = randn([B,Hkv,N,d])
  optionally q[:, 0] *= q_head0_scale (a power of two, so exact in bf16)
  each tensor is rounded to bf16 with round-to-nearest-even.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    N: int
    d: int
    causal: bool
    window: int
    seed: int
    q_head0_scale: float = 1.0
    note: str = ""

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def group(self) -> int:
        return self.Hq // self.Hkv


# The five workload shapes: a tiny bidirectional case, a ViT-Base-shaped
# short-sequence case, a GPT-2-small-shaped causal case with a sharpened head, a
# grouped-query causal long case and a causal sliding-window long case.
WORKLOADS = {
    "tiny": Workload("tiny", 1, 1, 1, 128, 64, False, 0, 0,
                     note="B1 H1 N128 d64 bidirectional"),
    "vit_base": Workload("vit_base", 256, 12, 12, 197, 64, False, 0, 1,
                         note="B256 H12 N197 d64 bidirectional (196 patches + class token)"),
    "gpt2_small": Workload("gpt2_small", 16, 12, 12, 1024, 64, True, 0, 2, 4.0,
                           note="B16 H12 N1024 d64 causal, Q x4 on head 0"),
    "gqa_8k": Workload("gqa_8k", 2, 32, 8, 8192, 128, True, 0, 3,
                       note="B2 Hq32 Hkv8 N8192 d128 causal"),
    "swa_16k": Workload("swa_16k", 2, 16, 16, 16384, 128, True, 1024, 4,
                        note="B2 H16 N16384 d128 causal, window 1024"),
}


def make_qkv(B: int, Hq: int, Hkv: int, N: int, d: int, seed: int,
             q_head0_scale: float = 1.0):
    """Return (q, k, v) as contiguous CPU bf16 tensors drawn from `seed`."""
    g = torch.Generator().manual_seed(int(seed))
    q = torch.randn((B, Hq, N, d), generator=g, dtype=torch.float32)
    k = torch.randn((B, Hkv, N, d), generator=g, dtype=torch.float32)
    v = torch.randn((B, Hkv, N, d), generator=g, dtype=torch.float32)
    if q_head0_scale != 1.0:
        q[:, 0] *= q_head0_scale
    return (q.to(torch.bfloat16).contiguous(), k.to(torch.bfloat16).contiguous(),
            v.to(torch.bfloat16).contiguous())


def make_workload(w: Workload):
    return make_qkv(w.B, w.Hq, w.Hkv, w.N, w.d, w.seed, w.q_head0_scale)


@dataclass(frozen=True)
class DecodeWorkload:
    """Nq queries per head at the end of an Nk-token sequence (key-value cache read)."""
    name: str
    B: int
    Hq: int
    Hkv: int
    Nq: int
    Nk: int
    d: int
    causal: bool
    seed: int
    note: str = ""

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


# A decode step of the GQA configuration's head layout: one new token per sequence
# reading an 8192-token cache (memory-bound: every key and value is read once).
DECODE_WORKLOADS = {
    "decode_8k": DecodeWorkload("decode_8k", 8, 32, 8, 1, 8192, 128, True, 6,
                                note="B8 Hq32 Hkv8 Nq1 Nk8192 d128 causal (decode step)"),
}


def make_qkv_decode(B: int, Hq: int, Hkv: int, Nq: int, Nk: int, d: int, seed: int):
    """(q [B,Hq,Nq,d], k [B,Hkv,Nk,d], v [B,Hkv,Nk,d]) as CPU bf16, drawn in that order
    from one generator seeded with `seed`, N(0,1) rounded to bf16."""
    g = torch.Generator().manual_seed(int(seed))
    q = torch.randn((B, Hq, Nq, d), generator=g, dtype=torch.float32)
    k = torch.randn((B, Hkv, Nk, d), generator=g, dtype=torch.float32)
    v = torch.randn((B, Hkv, Nk, d), generator=g, dtype=torch.float32)
    return (q.to(torch.bfloat16).contiguous(), k.to(torch.bfloat16).contiguous(),
            v.to(torch.bfloat16).contiguous())


def make_dout(B: int, Hq: int, N: int, d: int, seed: int):
    """Upstream gradient dO [B,Hq,N,d] for the backward pass: CPU bf16, N(0,1) from a
    generator seeded with `seed`, rounded to bf16."""
    g = torch.Generator().manual_seed(int(seed))
    return torch.randn((B, Hq, N, d), generator=g, dtype=torch.float32).to(torch.bfloat16).contiguous()


def make_signs(d: int, seed: int):
    """Random signs for incoherent processing: d values, each +1 or -1 with probability
    1/2, from a generator seeded with `seed` (as fp64 numpy)."""
    import numpy as np
    g = torch.Generator().manual_seed(int(seed))
    bits = torch.randint(0, 2, (d,), generator=g)
    return np.where(bits.numpy() == 1, -1.0, 1.0)
