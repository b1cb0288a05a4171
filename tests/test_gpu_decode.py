"""GPU parity of the packed-row (decode / split-KV) path against the oracle.

A call whose query rows of one KV group fit one 128-row tile (group * Tq <=
128: decode steps, short chunks) runs with the group's heads packed as rows,
and a long key range is split over the CTAs of a cluster whose partial
(m, l, O) are merged with the online-softmax rescale ("FlashAttention forward
in C", section 5: split-KV as in Flash-Decoding).  Every output row is
compared with the float64 oracle under the bf16 tolerances.
"""
import numpy as np
import pytest
import torch

import workloads
from parity import compare, gpu_attention, oracle_attention

pytestmark = pytest.mark.gpu

BF = torch.bfloat16


def _check(B, Hq, Hkv, Tq, Tk, d, seed, ctx, **kw):
    q, k, v = workloads.qkv(seed, B, Hq, Hkv, Tq, Tk, d, BF)
    o, lse = gpu_attention(q, k, v, **kw)
    eo, el = oracle_attention(q, k, v, **kw)
    compare(o, lse, eo, el, BF, ctx)
    return o, lse


@pytest.mark.parametrize("name", sorted(workloads.DECODE))
def test_decode_workloads(name):
    w = workloads.DECODE[name]
    p = w.problem
    _check(p.B, p.Hq, p.Hkv, p.Tq, p.Tk, p.d, w.seeds[0], name, scale=p.sm_scale, q_offset=p.q_offset, causal=True)


@pytest.mark.parametrize("Tk", [1, 2, 127, 128, 129, 383, 384, 385, 1000, 4097])
def test_decode_key_lengths(Tk):
    # split counts from 1 (fewer than 4 tiles) to 16, ragged last tiles
    _check(1, 8, 2, 1, Tk, 64, 300 + Tk, f"decode Tk={Tk}", scale=0.125, q_offset=Tk - 1, causal=True)


def test_decode_sinks_split():
    # the sink joins the sum once although the key range is split 16 ways
    B, Hq, Hkv, Tk, d = 2, 16, 8, 8192, 128
    z = workloads.sinks(41, Hq)
    _check(B, Hq, Hkv, 1, Tk, d, 40, "decode sinks split", scale=d ** -0.5, q_offset=Tk - 1, causal=True, sinks=z)
    # weights sum to 1 - p_sink with V = 1
    q, k, _ = workloads.qkv(40, B, Hq, Hkv, 1, Tk, d, BF)
    ones = torch.ones((B, Hkv, Tk, d), dtype=BF)
    o, lse = gpu_attention(q, k, ones, scale=d ** -0.5, q_offset=Tk - 1, causal=True, sinks=z)
    psink = torch.exp(z.double().view(1, -1, 1) - lse.double())
    assert (o.double() - (1.0 - psink)[..., None]).abs().max().item() <= 8e-3


def test_decode_window_split():
    # a window inside a long key range: the first splits see nothing
    _check(1, 32, 4, 1, 20000, 64, 42, "decode window", scale=0.125, q_offset=19999, causal=True, window=1500)


def test_decode_multi_token():
    # 4 new tokens per step (group 8 -> 32 packed rows), causal among them
    _check(2, 32, 4, 4, 5000, 128, 43, "decode 4 tokens", scale=128 ** -0.5, q_offset=4996, causal=True)


def test_decode_mask():
    B, Hq, Hkv, Tq, Tk = 2, 8, 2, 2, 1500
    g = torch.Generator().manual_seed(44)
    mask = torch.randn((B, Hq, Tq, Tk), generator=g)
    mask[torch.rand((B, Hq, Tq, Tk), generator=g) < 0.3] = -float("inf")
    mask[1, 3, 0, :] = -float("inf")  # one fully masked row: zeros, lse = -inf
    strides = (Hq * Tq * Tk, Tq * Tk, Tk, 1)
    o, lse = _check(B, Hq, Hkv, Tq, Tk, 96, 45, "decode mask", scale=0.1, q_offset=Tk - 2, causal=True, mask=mask,
                    mask_strides=strides)
    assert torch.isneginf(lse[1, 3, 0]) and torch.all(o[1, 3, 0] == 0)


def test_decode_no_keys_visible():
    # q_offset before the window's reach: no visible key, with and without a sink
    z = workloads.sinks(46, 8)
    q, k, v = workloads.qkv(46, 1, 8, 2, 1, 3000, 64, BF)
    o, lse = gpu_attention(q, k, v, scale=0.125, q_offset=5000, causal=True, window=100)
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))
    o, lse = gpu_attention(q, k, v, scale=0.125, q_offset=5000, causal=True, window=100, sinks=z)
    assert torch.all(o == 0)
    assert torch.allclose(lse, z.view(1, 8, 1), rtol=0, atol=1e-6)


def test_decode_noncausal_short_chunk():
    _check(1, 12, 3, 5, 700, 128, 47, "non-causal 5 rows", scale=0.09, causal=False)


def test_decode_split_matches_chunk_of_prefill():
    # The same rows through a prefill call and one decode call per row agree
    # within rounding (the split merge changes the summation order).
    T = 3000
    q, k, v = workloads.qkv(48, 1, 16, 8, T, T, 128, BF)
    o1, l1 = gpu_attention(q, k, v, scale=128 ** -0.5, causal=True)
    for r in (0, 1500, 2999):
        o, l = gpu_attention(q[:, :, r:r + 1].contiguous(), k[:, :, :r + 1].contiguous(), v[:, :, :r + 1].contiguous(),
                             scale=128 ** -0.5, q_offset=r, causal=True)
        assert (o.float() - o1[:, :, r:r + 1].float()).abs().max().item() <= 1e-2
        assert (l - l1[:, :, r:r + 1]).abs().max().item() <= 1e-3
