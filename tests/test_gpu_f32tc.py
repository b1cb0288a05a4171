"""GPU parity of the fp32 tensor-core path (FA_DTYPE_F32_TC: three TF32
products per matrix product) against the float64 oracle, at the fp32
tolerance (max |o - oracle| <= 1e-4, max |lse - oracle| <= 1e-4).

The same workloads as the SIMT fp32 path, tile edges on both sides of the
128-row query tile and the 32-key tile, every flag combination, strided
layouts, and the chunk invariance that "FlashAttention forward in C"
(section 2.4) asks of a q_offset chunk against the single call.
"""
import math

import numpy as np
import pytest
import torch

import exact_tiled_attention_flashattention_gb300 as fa
import workloads
from parity import compare, gpu_attention, oracle_attention, sample_rows

pytestmark = pytest.mark.gpu

F32 = torch.float32


def _run_and_compare(q, k, v, ctx, rows=None, **kw):
    o, lse = gpu_attention(q, k, v, fp32_tc=True, **kw)
    eo, el = oracle_attention(q, k, v, rows=rows, **kw)
    if rows is not None:
        o, lse = o[:, :, rows], lse[:, :, rows]
    return compare(o, lse, eo, el, F32, ctx)


def test_tile_crossing_d64():
    p = workloads.CONFIGS["tile_crossing_d64"].problem
    q, k, v = workloads.qkv(0, p.B, p.Hq, p.Hkv, p.Tq, p.Tk, p.d, F32)
    _run_and_compare(q, k, v, "tile_crossing", scale=1.0 / 8.0, causal=True)


def test_prefill511_28_layers():
    p = workloads.CONFIGS["prefill511_gqa16x8_d128_x28"].problem
    rows = np.arange(0, p.Tq, 7, dtype=np.int64)
    for layer in range(28):
        q, k, v = workloads.qkv(layer, p.B, p.Hq, p.Hkv, p.Tq, p.Tk, p.d, F32)
        full = layer in (0, 27)
        _run_and_compare(q, k, v, f"prefill511 layer {layer}", rows=None if full else rows, scale=p.sm_scale,
                         causal=True)


@pytest.mark.parametrize("name", ["longctx2044_gqa16x8_d128", "longctx8192_gqa16x8_d128"])
def test_long_context(name):
    w = workloads.CONFIGS[name]
    p = w.problem
    q, k, v = workloads.qkv(w.seeds[0], p.B, p.Hq, p.Hkv, p.Tq, p.Tk, p.d, F32)
    rows = None if p.Tq <= 2044 else sample_rows(p.Tq)
    _run_and_compare(q, k, v, name, rows=rows, scale=p.sm_scale, causal=True)


def test_window_sinks_chunked():
    w = workloads.CONFIGS["window128_sinks_gqa32x4_d64_chunked"]
    p = w.problem
    q, k, v = workloads.qkv(w.seeds[0], p.B, p.Hq, p.Hkv, p.Tq, p.Tk, p.d, F32)
    z = workloads.sinks(w.extra["sink_seed"], p.Hq)
    outs, lses = [], []
    for start, n in workloads.chunk_ranges(p.Tq, w.extra["chunk"]):
        o, lse = gpu_attention(q[:, :, start:start + n].contiguous(), k[:, :, :start + n].contiguous(),
                               v[:, :, :start + n].contiguous(), scale=p.sm_scale, q_offset=start, causal=True,
                               window=p.window, sinks=z, fp32_tc=True)
        outs.append(o)
        lses.append(lse)
    oc, lc = torch.cat(outs, dim=2), torch.cat(lses, dim=2)
    eo, el = oracle_attention(q, k, v, scale=p.sm_scale, causal=True, window=p.window, sinks=z)
    compare(oc, lc, eo, el, F32, "window/sinks chunked")
    o1, l1 = gpu_attention(q, k, v, scale=p.sm_scale, causal=True, window=p.window, sinks=z, fp32_tc=True)
    assert torch.equal(o1, oc), "chunked o differs from the single call"
    assert torch.equal(l1, lc), "chunked lse differs from the single call"


def test_mask_batch_d96():
    w = workloads.CONFIGS["mask_b4h8_t1024_d96"]
    p = w.problem
    q, k, v = workloads.qkv(w.seeds[0], p.B, p.Hq, p.Hkv, p.Tq, p.Tk, p.d, F32)
    m = workloads.strided_mask(w.extra["mask_seed"], p.Tq, p.Tk)
    strides = (0, 0, p.Tk, 1)
    o, lse = gpu_attention(q, k, v, scale=p.sm_scale, causal=False, mask=m, mask_strides=strides, fp32_tc=True)
    eo, el = oracle_attention(q, k, v, scale=p.sm_scale, causal=False, mask=m, mask_strides=strides)
    compare(o, lse, eo, el, F32, "mask batch")
    empty_rows = [0, 63, 64, 127, 500, 511, 512, 1023]
    assert torch.all(torch.isneginf(lse[:, :, empty_rows]))
    assert torch.all(o[:, :, empty_rows] == 0)


EDGE_T = [1, 2, 31, 32, 33, 63, 64, 65, 127, 128, 129, 130, 255, 257]


@pytest.mark.parametrize("d", [4, 36, 64, 100, 128])
def test_edges(d):
    for T in EDGE_T:
        q, k, v = workloads.qkv(T + d, 1, 2, 1, T, T, d, F32)
        _run_and_compare(q, k, v, f"edge T={T} d={d}", scale=1 / math.sqrt(d), causal=True)


FLAG_CASES = [
    # (Hq, Hkv, Tq, Tk, causal, window, q_offset, sinks, mask)
    (6, 2, 37, 37, True, 0, 0, False, False),
    (6, 1, 37, 37, True, 0, 0, False, False),
    (4, 2, 13, 37, True, 0, 24, False, False),
    (4, 2, 37, 37, True, 6, 0, False, False),
    (4, 2, 37, 37, False, 6, 0, False, False),
    (4, 4, 200, 300, False, 0, 0, False, False),
    (4, 2, 150, 300, True, 0, 150, True, False),
    (4, 2, 150, 300, True, 50, 150, True, True),
    (2, 1, 1, 300, True, 0, 299, False, False),
    (2, 1, 5, 3, True, 2, 10, False, False),
    (2, 1, 5, 3, True, 2, 10, True, False),
    (2, 2, 300, 140, False, 0, 0, False, True),
]


@pytest.mark.parametrize("case", FLAG_CASES, ids=[str(i) for i in range(len(FLAG_CASES))])
def test_flags(case):
    Hq, Hkv, Tq, Tk, causal, window, q_offset, use_sink, use_mask = case
    d = 64
    q, k, v = workloads.qkv(17, 2, Hq, Hkv, Tq, Tk, d, F32)
    z = workloads.sinks(3, Hq) if use_sink else None
    mask = strides = None
    if use_mask:
        g = torch.Generator().manual_seed(5)
        mask = torch.randn((2, Hq, Tq, Tk), generator=g)
        mask[torch.rand((2, Hq, Tq, Tk), generator=g) < 0.2] = -math.inf
        strides = (Hq * Tq * Tk, Tq * Tk, Tk, 1)
    _run_and_compare(q, k, v, f"flags {case}", scale=0.125, causal=causal, window=window, q_offset=q_offset,
                     sinks=z, mask=mask, mask_strides=strides or (0, 0, 0, 0))


@pytest.mark.parametrize("scale", [0.0, -0.125])
def test_non_positive_scale(scale):
    # scale <= 0 flips the order of the logits; the running maximum must
    # follow the scaled logits, not the raw products.
    q, k, v = workloads.qkv(23, 1, 2, 1, 70, 70, 64, F32)
    _run_and_compare(q, k, v, f"scale {scale}", scale=scale, causal=True)


def test_no_keys():
    q, _, _ = workloads.qkv(1, 1, 4, 2, 9, 0, 64, F32)
    kz = torch.zeros((1, 2, 0, 64), dtype=F32)
    o, lse = gpu_attention(q, kz, kz, scale=0.125, causal=False, fp32_tc=True)
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))
    z = workloads.sinks(2, 4)
    o, lse = gpu_attention(q, kz, kz, scale=0.125, causal=False, sinks=z, fp32_tc=True)
    assert torch.all(o == 0)
    assert torch.allclose(lse, z.view(1, 4, 1).expand_as(lse), rtol=0, atol=1e-6)


def test_strided_bshd_and_strided_out():
    # q, k, v read from [B, T, H, d] buffers, o written into a [B, T, H, d]
    # buffer with a padded row: the strided call equals the contiguous one
    # bit for bit.
    B, T, Hq, Hkv, d = 2, 300, 4, 2, 64
    g = torch.Generator().manual_seed(11)
    dev = torch.device("cuda", 0)
    qb = torch.randn((B, T, Hq, d), generator=g).to(dev)
    kb = torch.randn((B, T, Hkv, d), generator=g).to(dev)
    vb = torch.randn((B, T, Hkv, d), generator=g).to(dev)
    q, k, v = qb.transpose(1, 2), kb.transpose(1, 2), vb.transpose(1, 2)
    ob = torch.full((B, T, Hq, d + 8), float("nan"), device=dev)
    out = ob[..., :d].transpose(1, 2)
    o1, l1 = fa.attention(q, k, v, scale=0.125, causal=True, out=out, fp32_tc=True)
    o2, l2 = fa.attention(q.contiguous(), k.contiguous(), v.contiguous(), scale=0.125, causal=True, fp32_tc=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.all(torch.isnan(ob[..., d:])), "padding columns must stay untouched"
    eo, el = oracle_attention(q.cpu(), k.cpu(), v.cpu(), scale=0.125, causal=True)
    compare(o2.cpu(), l2.cpu(), eo, el, F32, "strided")


def test_sharp_logits():
    # Logits four times wider than the workloads' (a sharper softmax): one
    # TF32 product per matrix product (~1e-3 relative on each product) would
    # miss the fp32 tolerance by far; the split products must stay within it.
    q, k, v = workloads.qkv(29, 1, 2, 1, 256, 256, 128, F32)
    _run_and_compare(q * 4.0, k, v, "sharp logits", scale=1 / math.sqrt(128), causal=True)
