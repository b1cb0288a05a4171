"""GPU parity of the e4m3 path (FA_DTYPE_FP8_E4M3: e4m3 Q, K, V on
kind::f8f6f4 MMAs, P rounded to e4m3, bf16 O) against the float64 oracle on
the same e4m3 values.

The tolerance comes from the arithmetic (see parity.compare_fp8): every
element within 2^-4 max|v| + 2^-8 |o| of the oracle, lse within 1e-4; on
the workloads mean |do| <= 5e-3, and on the causal prefills max |do| <= 6e-2
(twice what a float64 simulation of the kernel's rounding gives there).
"""
import math

import numpy as np
import pytest
import torch

import exact_tiled_attention_flashattention_gb300 as fa
import workloads
from parity import compare_fp8, gpu_attention, oracle_attention, sample_rows

pytestmark = pytest.mark.gpu

F8 = torch.float8_e4m3fn


def _run(q, k, v, ctx, rows=None, causal_prefill=False, **kw):
    o, lse = gpu_attention(q, k, v, **kw)
    assert o.dtype == torch.bfloat16
    eo, el = oracle_attention(q, k, v, rows=rows, **kw)
    if rows is not None:
        o, lse = o[:, :, rows], lse[:, :, rows]
    return compare_fp8(o, lse, eo, el, v, q.shape[1] // k.shape[1], ctx, causal_prefill=causal_prefill)


def test_prefill511_28_layers():
    p = workloads.CONFIGS["prefill511_gqa16x8_d128_x28"].problem
    rows = np.arange(0, p.Tq, 7, dtype=np.int64)
    for layer in range(28):
        q, k, v = workloads.qkv(layer, p.B, p.Hq, p.Hkv, p.Tq, p.Tk, p.d, F8)
        full = layer in (0, 27)
        _run(q, k, v, f"prefill511 e4m3 layer {layer}", rows=None if full else rows, causal_prefill=True,
             scale=p.sm_scale, causal=True)


@pytest.mark.parametrize("name", ["longctx2044_gqa16x8_d128", "longctx8192_gqa16x8_d128"])
def test_long_context(name):
    w = workloads.CONFIGS[name]
    p = w.problem
    q, k, v = workloads.qkv(w.seeds[0], p.B, p.Hq, p.Hkv, p.Tq, p.Tk, p.d, F8)
    rows = None if p.Tq <= 2044 else sample_rows(p.Tq)
    _run(q, k, v, name, rows=rows, causal_prefill=True, scale=p.sm_scale, causal=True)


def test_window_sinks_chunked():
    w = workloads.CONFIGS["window128_sinks_gqa32x4_d64_chunked"]
    p = w.problem
    q, k, v = workloads.qkv(w.seeds[0], p.B, p.Hq, p.Hkv, p.Tq, p.Tk, p.d, F8)
    z = workloads.sinks(w.extra["sink_seed"], p.Hq)
    outs, lses = [], []
    for start, n in workloads.chunk_ranges(p.Tq, w.extra["chunk"]):
        o, lse = gpu_attention(q[:, :, start:start + n].contiguous(), k[:, :, :start + n].contiguous(),
                               v[:, :, :start + n].contiguous(), scale=p.sm_scale, q_offset=start, causal=True,
                               window=p.window, sinks=z)
        outs.append(o)
        lses.append(lse)
    oc, lc = torch.cat(outs, dim=2), torch.cat(lses, dim=2)
    eo, el = oracle_attention(q, k, v, scale=p.sm_scale, causal=True, window=p.window, sinks=z)
    compare_fp8(oc, lc, eo, el, v, p.Hq // p.Hkv, "window/sinks chunked", workload=True)
    # Absolute key tiles: the chunked calls equal the single call bit for bit.
    o1, l1 = gpu_attention(q, k, v, scale=p.sm_scale, causal=True, window=p.window, sinks=z)
    assert torch.equal(o1, oc) and torch.equal(l1, lc)


def test_mask_batch_d96():
    w = workloads.CONFIGS["mask_b4h8_t1024_d96"]
    p = w.problem
    q, k, v = workloads.qkv(w.seeds[0], p.B, p.Hq, p.Hkv, p.Tq, p.Tk, p.d, F8)
    m = workloads.strided_mask(w.extra["mask_seed"], p.Tq, p.Tk)
    strides = (0, 0, p.Tk, 1)
    rows = np.arange(0, p.Tq, 5, dtype=np.int64)
    o, lse = gpu_attention(q, k, v, scale=p.sm_scale, causal=False, mask=m, mask_strides=strides)
    eo, el = oracle_attention(q, k, v, rows=rows, scale=p.sm_scale, causal=False, mask=m, mask_strides=strides)
    compare_fp8(o[:, :, rows], lse[:, :, rows], eo, el, v, 1, "mask batch e4m3 d96", workload=True)
    empty_rows = [0, 63, 64, 127, 500, 511, 512, 1023]
    assert torch.all(torch.isneginf(lse[:, :, empty_rows]))
    assert torch.all(o[:, :, empty_rows] == 0)


EDGE_T = [1, 2, 63, 64, 65, 127, 128, 129, 130, 255, 257]


@pytest.mark.parametrize("d", [16, 64, 96, 128])
def test_edges(d):
    for T in EDGE_T:
        q, k, v = workloads.qkv(T + d, 1, 2, 1, T, T, d, F8)
        _run(q, k, v, f"edge e4m3 T={T} d={d}", scale=1 / math.sqrt(d), causal=True)


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
    q, k, v = workloads.qkv(17, 2, Hq, Hkv, Tq, Tk, 64, F8)
    z = workloads.sinks(3, Hq) if use_sink else None
    mask = strides = None
    if use_mask:
        g = torch.Generator().manual_seed(5)
        mask = torch.randn((2, Hq, Tq, Tk), generator=g)
        mask[torch.rand((2, Hq, Tq, Tk), generator=g) < 0.2] = -math.inf
        strides = (Hq * Tq * Tk, Tq * Tk, Tk, 1)
    _run(q, k, v, f"flags {case}", scale=0.125, causal=causal, window=window, q_offset=q_offset, sinks=z,
         mask=mask, mask_strides=strides or (0, 0, 0, 0))


def test_no_keys():
    q, _, _ = workloads.qkv(1, 1, 4, 2, 9, 0, 64, F8)
    kz = torch.zeros((1, 2, 0, 64), dtype=F8)
    o, lse = gpu_attention(q, kz, kz, scale=0.125, causal=False)
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))
    z = workloads.sinks(2, 4)
    o, lse = gpu_attention(q, kz, kz, scale=0.125, causal=False, sinks=z)
    assert torch.all(o == 0)
    assert torch.allclose(lse, z.view(1, 4, 1).expand_as(lse), rtol=0, atol=1e-6)


def test_one_key_is_exact():
    # A row that sees one key gets p = 1 exactly: o = v_0 rounded to bf16.
    q, k, v = workloads.qkv(5, 1, 2, 1, 1, 1, 128, F8)
    o, lse = gpu_attention(q, k, v, scale=0.1, causal=True)
    assert torch.equal(o[0, :, 0], v[0, 0, 0].float().to(torch.bfloat16).expand(2, -1))


def test_strided_bshd_and_strided_out():
    B, T, Hq, Hkv, d = 2, 300, 4, 2, 64
    dev = torch.device("cuda", 0)
    g = torch.Generator().manual_seed(11)
    qb = torch.randn((B, T, Hq, d), generator=g).to(F8).to(dev)
    kb = torch.randn((B, T, Hkv, d), generator=g).to(F8).to(dev)
    vb = torch.randn((B, T, Hkv, d), generator=g).to(F8).to(dev)
    q, k, v = qb.transpose(1, 2), kb.transpose(1, 2), vb.transpose(1, 2)
    ob = torch.full((B, T, Hq, d + 8), float("nan"), dtype=torch.bfloat16, device=dev)
    out = ob[..., :d].transpose(1, 2)
    o1, l1 = fa.attention(q, k, v, scale=0.125, causal=True, out=out)
    o2, l2 = fa.attention(q.contiguous(), k.contiguous(), v.contiguous(), scale=0.125, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.all(torch.isnan(ob[..., d:]))
    eo, el = oracle_attention(q.cpu(), k.cpu(), v.cpu(), scale=0.125, causal=True)
    compare_fp8(o2.cpu(), l2.cpu(), eo, el, v.cpu(), Hq // Hkv, "strided e4m3")
