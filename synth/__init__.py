"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic.  Both the CUDA path and the CPU oracle consume exactly
the tensors produced here, so an input never comes from either side.

Workloads (sizes, distributions) follow the handbook chapter "Context
parallelism: Ring Attention and Ulysses" (section "Which operations partition
directly": ``make_qkv`` draws q, k, v ~ N(0, 1) of shape [S, H, D] after
``torch.manual_seed(0)``) and the packed-document workload of the MaxText pull
request "Add Packing Support for Context Parallelism (Ring Attention) #2906"
(documents packed into one stream, block-diagonal causal mask).
"""
from __future__ import annotations

import numpy as np
import torch

__all__ = [
    "make_qkv",
    "make_inputs",
    "doc_lengths",
    "cu_seqlens_from_lengths",
    "WORKLOADS",
]


def make_qkv(S: int = 32, H: int = 8, D: int = 16):
    """The handbook's test data: global seed 0, then three ``randn(S, H, D)``
    draws in the order q, k, v (fp32, CPU)."""
    torch.manual_seed(0)
    return torch.randn(S, H, D), torch.randn(S, H, D), torch.randn(S, H, D)


def make_inputs(S: int, Hq: int, Hkv: int, D: int, dtype: torch.dtype = torch.bfloat16,
                seed: int = 0, with_dout: bool = False):
    """q [S,Hq,D], k/v [S,Hkv,D] (and dO [S,Hq,D] when ``with_dout``), N(0,1).

    Drawn in fp32 on the CPU from ``torch.Generator().manual_seed(seed)`` in the
    order q, k, v, dO, then cast (round-to-nearest-even) to ``dtype``.  The cast
    tensors are the exact values both the GPU and the oracle see.
    """
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(S, Hq, D, generator=g)
    k = torch.randn(S, Hkv, D, generator=g)
    v = torch.randn(S, Hkv, D, generator=g)
    out = [q.to(dtype), k.to(dtype), v.to(dtype)]
    if with_dout:
        out.append(torch.randn(S, Hq, D, generator=g).to(dtype))
    return tuple(out)


def doc_lengths(S: int, lo: int = 512, hi: int = 16384, seed: int = 0) -> list[int]:
    """Document lengths for a packed stream of S tokens.

    Lengths are drawn i.i.d. uniform on [lo, hi] (``randint(lo, hi + 1)`` from
    ``torch.Generator().manual_seed(seed)``) while the running total is below S;
    the last draw is cut so the lengths sum to exactly S.
    """
    g = torch.Generator().manual_seed(seed)
    out: list[int] = []
    total = 0
    while total < S:
        L = int(torch.randint(lo, hi + 1, (1,), generator=g).item())
        L = min(L, S - total)
        out.append(L)
        total += L
    return out


def cu_seqlens_from_lengths(lengths) -> np.ndarray:
    """Prefix sums [0, L0, L0+L1, ..., S] as int32 (the packed-stream boundaries)."""
    cu = np.zeros(len(lengths) + 1, dtype=np.int64)
    cu[1:] = np.cumsum(np.asarray(lengths, dtype=np.int64))
    return cu.astype(np.int32)


# The five workloads the library is exercised on (sizes only; no arithmetic).
WORKLOADS = {
    "tiny_exact_s32_h8_d16_fp32_p4": dict(S=32, Hq=8, Hkv=8, D=16, dtype="f32", P=4),
    "ring_fwd_mha_s8192_h32_d128_bf16_p8_zigzag": dict(S=8192, Hq=32, Hkv=32, D=128, dtype="bf16", P=8),
    "ulysses_fwd_s32768_h32_d128_bf16_p16": dict(S=32768, Hq=32, Hkv=32, D=128, dtype="bf16", P=16),
    "gqa_ring_fwd_bwd_s65536_hq32_hkv8_d128_bf16_p4_zigzag": dict(S=65536, Hq=32, Hkv=8, D=128, dtype="bf16", P=4),
    "packed_varlen_s131072_hq32_hkv8_d128_bf16_p8": dict(S=131072, Hq=32, Hkv=8, D=128, dtype="bf16", P=8),
}
