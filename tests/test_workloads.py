"""Host checks of the workload descriptions and the seeded input recipe.

The benchmark's metric counts 4*d FLOPs per visible (query row, key) pair
(the "causal-adjusted" count: Q.K^T and P.V each take 2*d per pair), so the
visible-pair count of ``workloads.Problem`` decides every reported TFLOP/s.
It is pinned here three independent ways: closed forms of the visibility rule
of "FlashAttention forward in C" (section 2.1, "What is computed"), brute
force over every (row, key) pair on small shapes, and the float64 oracle
itself, whose lse with q = 0 is ln |V_i| for every row (uniform weights over
the visible keys), so that sum_i exp(lse_i) is the pair count the oracle
sees.  The chunking of the 4096-token prompt (1000-token chunks with
q_offset) and the seeded generators are pinned as well.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from workloads import Problem


def _brute_pairs(Tq, Tk, causal, window, q_offset):
    """Visible pairs of one (batch, head), by testing every (i, j)."""
    n = 0
    for i in range(Tq):
        p = q_offset + i
        for j in range(Tk):
            if causal and j > p:
                continue
            if window > 0 and j <= p - window:
                continue
            n += 1
    return n


# --- closed forms ------------------------------------------------------------

def test_causal_square_is_triangular():
    for T in (1, 2, 127, 128, 129, 511, 2044):
        assert Problem(1, 1, 1, T, T, 64).visible_pairs() == T * (T + 1) // 2


def test_non_causal_is_full():
    assert Problem(4, 8, 8, 1024, 1024, 96, causal=False).visible_pairs() == 4 * 8 * 1024 * 1024
    assert Problem(1, 2, 1, 7, 13, 64, causal=False).visible_pairs() == 2 * 7 * 13


def test_causal_window_closed_form():
    # row p sees min(p + 1, w) keys: w(w+1)/2 over the first w rows, then w each
    for T, w in ((4096, 128), (300, 1), (300, 299), (300, 300), (300, 5000)):
        ww = min(w, T)
        assert Problem(1, 1, 1, T, T, 64, window=w).visible_pairs() == ww * (ww + 1) // 2 + (T - ww) * ww


def test_decode_step_sees_every_key():
    for Tk in (1, 328, 2044, 32768):
        assert Problem(1, 16, 8, 1, Tk, 128, q_offset=Tk - 1).visible_pairs() == 16 * Tk


def test_headline_flop_counts():
    # one 511-token layer: 16 heads x 511*512/2 pairs x 4*128 FLOPs
    p = workloads.CONFIGS["prefill511_gqa16x8_d128_x28"].problem
    assert p.flops() == 4 * 128 * 16 * (511 * 512 // 2) == 1_071_644_672
    for name, T in (("longctx2044_gqa16x8_d128", 2044), ("longctx8192_gqa16x8_d128", 8192),
                    ("longctx32768_gqa16x8_d128", 32768)):
        assert workloads.CONFIGS[name].problem.flops() == 4 * 128 * 16 * T * (T + 1) // 2
    assert workloads.CONFIGS["longctx32768_gqa16x8_d128"].problem.flops() == 4_398_180_728_832
    w = workloads.CONFIGS["mask_b4h8_t1024_d96"].problem
    assert w.flops() == 4 * 96 * 4 * 8 * 1024 * 1024  # dense: masked entries are not skipped


# --- brute force -------------------------------------------------------------

@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("window", [0, 1, 3, 6, 40])
@pytest.mark.parametrize("q_offset", [0, 1, 24])
@pytest.mark.parametrize("Tq,Tk", [(0, 5), (1, 1), (5, 5), (17, 37), (37, 17), (33, 60)])
def test_pairs_match_brute_force(causal, window, q_offset, Tq, Tk):
    p = Problem(2, 3, 1, Tq, Tk, 64, causal=causal, window=window, q_offset=q_offset)
    assert p.visible_pairs() == 2 * 3 * _brute_pairs(Tq, Tk, causal, window, q_offset)


# --- the oracle's own visibility ---------------------------------------------

@pytest.mark.parametrize("causal,window,q_offset,Tq,Tk", [
    (True, 0, 0, 45, 45), (True, 7, 0, 45, 45), (True, 7, 30, 20, 50),
    (False, 5, 3, 19, 40), (False, 0, 0, 9, 31), (True, 0, 60, 8, 40)])
def test_pairs_match_oracle_visibility(causal, window, q_offset, Tq, Tk):
    """q = 0 gives every visible key the weight 1/|V_i|, so lse_i = ln |V_i|
    (and -inf for an empty row)."""
    B, Hq, Hkv, d = 1, 4, 2, 8
    q = np.zeros((B, Hq, Tq, d))
    k = np.random.default_rng(1).standard_normal((B, Hkv, Tk, d))
    v = np.random.default_rng(2).standard_normal((B, Hkv, Tk, d))
    _, lse = oracle.attention(q, k, v, 0.125, q_offset=q_offset, causal=causal, window=window)
    per_row = np.where(np.isneginf(lse), 0.0, np.exp(lse))
    assert np.allclose(per_row, np.rint(per_row), atol=1e-9)
    p = Problem(B, Hq, Hkv, Tq, Tk, d, causal=causal, window=window, q_offset=q_offset)
    assert int(np.rint(per_row).sum()) == p.visible_pairs()


# --- chunked prefill ---------------------------------------------------------

def test_chunk_ranges_of_the_windowed_prompt():
    assert workloads.chunk_ranges(4096, 1000) == [(0, 1000), (1000, 1000), (2000, 1000), (3000, 1000),
                                                  (4000, 96)]
    assert workloads.chunk_ranges(0, 1000) == []
    assert workloads.chunk_ranges(1000, 1000) == [(0, 1000)]


def test_chunked_pairs_equal_one_call():
    """Each chunk is a call with Tq = its length, q_offset = its start and
    Tk = q_offset + Tq; the chunks together see exactly the pairs of one
    call over the whole prompt (516,160 per (batch, head) for w = 128)."""
    w = workloads.CONFIGS["window128_sinks_gqa32x4_d64_chunked"]
    p = w.problem
    whole = p.visible_pairs()
    parts = 0
    for s, n in workloads.chunk_ranges(p.Tq, w.extra["chunk"]):
        parts += Problem(p.B, p.Hq, p.Hkv, n, s + n, p.d, causal=True, window=p.window, q_offset=s).visible_pairs()
    assert parts == whole == p.B * p.Hq * 516_160


# --- seeded inputs -------------------------------------------------------------

def test_qkv_is_deterministic_and_seeded_per_tensor():
    a = workloads.qkv(3, 1, 4, 2, 33, 40, 16)
    b = workloads.qkv(3, 1, 4, 2, 33, 40, 16)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    c = workloads.qkv(4, 1, 4, 2, 33, 40, 16)
    assert not torch.equal(a[0], c[0])
    # Q, K and V come from generators 3*seed + 0, 1, 2: K of seed 3 is generator 10's draw
    assert a[2].shape == (1, 2, 40, 16) and a[0].shape == (1, 4, 33, 16)
    g = torch.Generator(device="cpu")
    g.manual_seed(3 * 3 + 1)
    assert torch.equal(a[1], torch.randn((1, 2, 40, 16), generator=g, dtype=torch.float32))


def test_bf16_inputs_are_the_rounded_fp32_draw():
    f = workloads.qkv(7, 1, 2, 1, 20, 20, 32, torch.float32)
    h = workloads.qkv(7, 1, 2, 1, 20, 20, 32, torch.bfloat16)
    for x, y in zip(f, h):
        assert y.dtype == torch.bfloat16
        assert torch.equal(x.to(torch.bfloat16), y)


def test_strided_mask_recipe():
    m = workloads.strided_mask(11, 1024, 1024)
    vals = m.unique()
    assert set(vals.tolist()) <= {0.0, -math.inf}
    full = (0, 63, 64, 127, 500, 511, 512, 1023)
    for r in full:
        assert torch.isneginf(m[r]).all()
    rest = torch.ones(1024, dtype=torch.bool)
    rest[list(full)] = False
    frac = torch.isneginf(m[rest]).double().mean().item()
    # 1016 * 1024 Bernoulli(0.1) draws: the standard deviation is 3e-4
    assert abs(frac - 0.1) < 3e-3
    # every other row keeps at least one visible key (so only the 8 rows are empty)
    assert (~torch.isneginf(m[rest])).any(dim=1).all()
