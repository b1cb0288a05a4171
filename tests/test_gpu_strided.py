"""Strided layouts through fa_fwd_strided (the binding passes a tensor's own
strides): [B, T, H, d] buffers seen as [B, H, T, d], a [T, H*d] buffer,
padded rows and a [B, T, H, d] output.  Only addressing differs from the
contiguous call, so results must match it bit for bit (and the oracle
within tolerance)."""
import pytest
import torch

import exact_tiled_attention_flashattention_gb300 as fa
import workloads
from parity import compare, oracle_attention

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "bf16": torch.bfloat16}
DEV = torch.device("cuda", 0)


def _contig(q, k, v, **kw):
    o, l = fa.attention(q.to(DEV), k.to(DEV), v.to(DEV), **kw)
    torch.cuda.synchronize()
    return o.cpu(), l.cpu()


def _bshd_view(t):
    """The same values stored as [B, T, H, d], seen as [B, H, T, d]."""
    return t.to(DEV).transpose(1, 2).contiguous().transpose(1, 2)


def _padded_view(t, pad):
    B, H, T, d = t.shape
    buf = torch.zeros((B, H, T, d + pad), dtype=t.dtype, device=DEV)
    buf[..., :d] = t.to(DEV)
    return buf[..., :d]


CASES = [
    # (B, Hq, Hkv, Tq, Tk, d, flags)  prefill and packed (decode-like) shapes
    (2, 8, 4, 300, 300, 64, dict(causal=True)),
    (1, 16, 8, 1, 2500, 128, dict(causal=True, q_offset=2499)),
    (2, 12, 3, 5, 900, 96, dict(causal=False)),
    (1, 4, 2, 200, 520, 128, dict(causal=True, q_offset=320, window=100)),
]


@pytest.mark.parametrize("dt", ["bf16", "f32"])
@pytest.mark.parametrize("case", CASES, ids=[str(i) for i in range(len(CASES))])
def test_bshd_inputs_and_output(dt, case):
    B, Hq, Hkv, Tq, Tk, d, flags = case
    q, k, v = workloads.qkv(60 + Tq, B, Hq, Hkv, Tq, Tk, d, DT[dt])
    kw = dict(scale=d ** -0.5, **flags)
    o_ref, l_ref = _contig(q, k, v, **kw)
    out = torch.empty((B, Tq, Hq, d), dtype=DT[dt], device=DEV).transpose(1, 2)  # [B, T, H, d] storage
    o, l = fa.attention(_bshd_view(q), _bshd_view(k), _bshd_view(v), out=out, **kw)
    torch.cuda.synchronize()
    assert o.data_ptr() == out.data_ptr()
    assert torch.equal(o.cpu(), o_ref) and torch.equal(l.cpu(), l_ref)
    eo, el = oracle_attention(q, k, v, **kw)
    compare(o.cpu(), l.cpu(), eo, el, DT[dt], f"bshd {case} {dt}")


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_seq_by_hd_layout(dt):
    # one [T, H*d] buffer per tensor (B = 1), as an engine keeps projections
    T, Hq, Hkv, d = 257, 8, 2, 64
    q, k, v = workloads.qkv(70, 1, Hq, Hkv, T, T, d, DT[dt])
    kw = dict(scale=0.125, causal=True)
    o_ref, l_ref = _contig(q, k, v, **kw)

    def as_2d(t):
        H = t.shape[1]
        flat = t[0].to(DEV).transpose(0, 1).reshape(T, H * d)  # [T, H*d]
        return flat.view(T, H, d).permute(1, 0, 2).unsqueeze(0)  # [1, H, T, d] view

    o, l = fa.attention(as_2d(q), as_2d(k), as_2d(v), **kw)
    torch.cuda.synchronize()
    assert torch.equal(o.cpu(), o_ref) and torch.equal(l.cpu(), l_ref)


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_padded_rows(dt):
    B, Hq, Hkv, Tq, Tk, d = 2, 4, 4, 150, 333, 64
    q, k, v = workloads.qkv(71, B, Hq, Hkv, Tq, Tk, d, DT[dt])
    kw = dict(scale=0.125, causal=False)
    o_ref, l_ref = _contig(q, k, v, **kw)
    o, l = fa.attention(_padded_view(q, 8), _padded_view(k, 24), _padded_view(v, 16), **kw)
    torch.cuda.synchronize()
    assert torch.equal(o.cpu(), o_ref) and torch.equal(l.cpu(), l_ref)


def test_strided_sinks_mask_bf16():
    B, Hq, Hkv, Tq, Tk, d = 2, 8, 2, 64, 700, 128
    q, k, v = workloads.qkv(72, B, Hq, Hkv, Tq, Tk, d, torch.bfloat16)
    z = workloads.sinks(73, Hq).to(DEV)
    g = torch.Generator().manual_seed(74)
    mask = torch.randn((Tq, Tk), generator=g)
    mask[torch.rand((Tq, Tk), generator=g) < 0.2] = -float("inf")
    md = mask.to(DEV)
    kw = dict(scale=d ** -0.5, causal=True, q_offset=Tk - Tq, sinks=z, mask=md, mask_strides=(0, 0, Tk, 1))
    o_ref, l_ref = _contig(q, k, v, **kw)
    o, l = fa.attention(_bshd_view(q), _bshd_view(k), _bshd_view(v), **kw)
    torch.cuda.synchronize()
    assert torch.equal(o.cpu(), o_ref) and torch.equal(l.cpu(), l_ref)
