"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle.

This module holds no attention arithmetic: it only draws tensors from seeded
CPU generators and describes the workload shapes.  Both the CUDA path and the
float64 oracle consume exactly the tensors made here (bf16 inputs are rounded
once, here, and the oracle widens the rounded values exactly).

Recipe: every Q/K/V tensor is ``torch.randn`` in float32 from a CPU
``torch.Generator`` seeded with ``3*seed + {0, 1, 2}`` for Q, K, V, then cast to
the compute dtype.  The workloads stand in for the pages' prompts and model
weights (a 511-token prompt through a 28-layer 16q/8kv d=128 model, a 2k
context, a windowed sink model fed in chunks), which are not available: only
their shapes are reproduced.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

__all__ = ["Problem", "qkv", "sinks", "strided_mask", "CONFIGS", "DECODE", "PAGED", "VARLEN", "paged_lengths", "chunk_ranges"]


@dataclass(frozen=True)
class Problem:
    """Shape and flags of one attention call (BHSD layout)."""
    B: int
    Hq: int
    Hkv: int
    Tq: int
    Tk: int
    d: int
    causal: bool = True
    window: int = 0
    q_offset: int = 0
    scale: float | None = None  # None: 1/sqrt(d)

    @property
    def sm_scale(self) -> float:
        return self.scale if self.scale is not None else 1.0 / math.sqrt(self.d)

    def visible_pairs(self) -> int:
        """Number of (query row, key) pairs the visibility rule admits, summed
        over batch and query heads (counts positions only; additive masks are
        not subtracted).  Used for causal-adjusted FLOP counts."""
        per_head = 0
        for i in range(self.Tq):
            p = self.q_offset + i
            hi = min(self.Tk, p + 1) if self.causal else self.Tk
            lo = max(0, p - self.window + 1) if self.window > 0 else 0
            per_head += max(0, hi - lo)
        return per_head * self.B * self.Hq

    def flops(self) -> int:
        """Causal-adjusted FLOPs: 4 * d per visible (row, key) pair (2 for
        Q.K^T, 2 for P.V)."""
        return 4 * self.d * self.visible_pairs()


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def qkv(seed: int, B: int, Hq: int, Hkv: int, Tq: int, Tk: int, d: int,
        dtype: torch.dtype = torch.float32):
    """Q [B,Hq,Tq,d], K and V [B,Hkv,Tk,d], iid N(0,1), CPU tensors of ``dtype``."""
    q = torch.randn((B, Hq, Tq, d), generator=_gen(3 * seed + 0), dtype=torch.float32)
    k = torch.randn((B, Hkv, Tk, d), generator=_gen(3 * seed + 1), dtype=torch.float32)
    v = torch.randn((B, Hkv, Tk, d), generator=_gen(3 * seed + 2), dtype=torch.float32)
    return q.to(dtype), k.to(dtype), v.to(dtype)


def sinks(seed: int, H: int) -> torch.Tensor:
    """One learned sink logit per query head, N(0,1), float32 [H]."""
    return torch.randn((H,), generator=_gen(seed), dtype=torch.float32)


def strided_mask(seed: int, Tq: int, Tk: int, p_neg_inf: float = 0.1,
                 full_rows=(0, 63, 64, 127, 500, 511, 512, 1023)) -> torch.Tensor:
    """Additive mask [Tq, Tk] float32: -inf with probability ``p_neg_inf``
    (iid), else 0; the rows in ``full_rows`` (those < Tq) are all -inf.  Used
    with strides (0, 0, Tk, 1): broadcast over batch and heads."""
    u = torch.rand((Tq, Tk), generator=_gen(seed), dtype=torch.float32)
    m = torch.zeros((Tq, Tk), dtype=torch.float32)
    m[u < p_neg_inf] = -math.inf
    for r in full_rows:
        if r < Tq:
            m[r, :] = -math.inf
    return m


def chunk_ranges(total: int, chunk: int):
    """[(start, length)] splitting a prompt of ``total`` tokens into chunks."""
    return [(s, min(chunk, total - s)) for s in range(0, total, chunk)]


@dataclass(frozen=True)
class Workload:
    name: str
    problem: Problem
    dtypes: tuple
    seeds: tuple = (0,)
    extra: dict = field(default_factory=dict)


# The five workloads: shapes of the pages' prefill runs, stated once here.
CONFIGS = {
    # 130 rows cross a 64-key tile boundary twice; scale 1/sqrt(64) = 1/8.
    "tile_crossing_d64": Workload(
        "tile_crossing_d64", Problem(1, 1, 1, 130, 130, 64, causal=True), ("f32",), seeds=(0,)),
    # 511-token prefill, 16 query heads on 8 KV heads, d=128, 28 layers.
    "prefill511_gqa16x8_d128_x28": Workload(
        "prefill511_gqa16x8_d128_x28", Problem(1, 16, 8, 511, 511, 128, causal=True),
        ("bf16", "f32"), seeds=tuple(range(28))),
    # long-context causal prefill, bf16.
    "longctx2044_gqa16x8_d128": Workload(
        "longctx2044_gqa16x8_d128", Problem(1, 16, 8, 2044, 2044, 128), ("bf16",), seeds=(100,)),
    "longctx8192_gqa16x8_d128": Workload(
        "longctx8192_gqa16x8_d128", Problem(1, 16, 8, 8192, 8192, 128), ("bf16",), seeds=(101,)),
    "longctx32768_gqa16x8_d128": Workload(
        "longctx32768_gqa16x8_d128", Problem(1, 16, 8, 32768, 32768, 128), ("bf16",), seeds=(102,)),
    # windowed GQA with sinks, 4096-token prompt fed as 1000-token chunks.
    "window128_sinks_gqa32x4_d64_chunked": Workload(
        "window128_sinks_gqa32x4_d64_chunked", Problem(2, 32, 4, 4096, 4096, 64, causal=True, window=128),
        ("bf16", "f32"), seeds=(4,), extra={"chunk": 1000, "sink_seed": 7}),
    # additive-mask batch, broadcast strided mask with 10% -inf and 8 empty rows.
    "mask_b4h8_t1024_d96": Workload(
        "mask_b4h8_t1024_d96", Problem(4, 8, 8, 1024, 1024, 96, causal=False),
        ("f32",), seeds=(5,), extra={"mask_seed": 11}),
}


# Decode steps (one new token per sequence: Tq = 1 at q_offset = Tk - 1, causal),
# "FlashAttention forward in C" section 2.1: the same flags serve a decode
# step.  Geometries: the 16q/8kv d=128 model of the prefill configurations at
# its three context lengths, a batch of 8 such sequences, and the 9q/3kv d=64
# model of the CPU flash-attention page after a 128-token prefill and 200
# decode steps.  These are not among the benchmark's headline configurations;
# they measure the split-KV decode path.
DECODE = {
    "decode_gqa16x8_d128_k2044": Workload(
        "decode_gqa16x8_d128_k2044", Problem(1, 16, 8, 1, 2044, 128, q_offset=2043), ("bf16",), seeds=(200,)),
    "decode_gqa16x8_d128_k8192": Workload(
        "decode_gqa16x8_d128_k8192", Problem(1, 16, 8, 1, 8192, 128, q_offset=8191), ("bf16",), seeds=(201,)),
    "decode_gqa16x8_d128_k32768": Workload(
        "decode_gqa16x8_d128_k32768", Problem(1, 16, 8, 1, 32768, 128, q_offset=32767), ("bf16",), seeds=(202,)),
    "decode_b8_gqa16x8_d128_k8192": Workload(
        "decode_b8_gqa16x8_d128_k8192", Problem(8, 16, 8, 1, 8192, 128, q_offset=8191), ("bf16",), seeds=(203,)),
    "decode_gqa9x3_d64_k328": Workload(
        "decode_gqa9x3_d64_k328", Problem(1, 9, 3, 1, 328, 64, q_offset=327), ("bf16",), seeds=(204,)),
}


def paged_lengths(seed: int, B: int, lo: int, hi: int) -> list:
    """Per-sequence cache lengths, uniform in [lo, hi] (seeded)."""
    g = _gen(seed)
    return [int(x) for x in torch.randint(lo, hi + 1, (B,), generator=g)]


# Paged decode steps (one new token per sequence over a paged cache): 8 and 32
# sequences of the 16q/8kv d=128 model with lengths drawn in [4096, 8192],
# 64-token pages.
PAGED = {
    "paged_b8_gqa16x8_d128_k4k-8k_p64": dict(B=8, Hq=16, Hkv=8, d=128, lo=4096, hi=8192, page_size=64, seed=210),
    "paged_b32_gqa16x8_d128_k4k-8k_p64": dict(B=32, Hq=16, Hkv=8, d=128, lo=4096, hi=8192, page_size=64, seed=211),
}


# A variable-length prefill batch: 8 prompts of the 16q/8kv d=128 model with
# lengths drawn in [256, 4096] (causal, each its own sequence).
VARLEN = {
    "varlen_b8_gqa16x8_d128_256-4096": dict(B=8, Hq=16, Hkv=8, d=128, lo=256, hi=4096, seed=220),
}
