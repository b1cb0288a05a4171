"""GPU parity of split-KV decode through a caller-owned workspace.

fa_fwd_splitkv splits each (batch, KV head) of a packed-row call over as many
CTAs as fill the SMs (Flash-Decoding, named on "FlashAttention forward in C",
section 5: long contexts split across thread blocks, the partial (m, l, a)
merged with the same rescale).  The partials go through global memory and the
last CTA of a KV head to finish merges them.  Every output row is compared
with the float64 oracle under the bf16 tolerances; the merge takes the
partials in split order, so repeated calls agree bit for bit.
"""
import pytest
import torch

import exact_tiled_attention_flashattention_gb300 as fa
import workloads
from parity import compare, gpu_attention, oracle_attention

pytestmark = pytest.mark.gpu

BF = torch.bfloat16


def splitkv(q, k, v, *, workspace=None, **kw):
    dev = torch.device("cuda", 0)
    qd, kd, vd = (x.to(dev).contiguous() for x in (q, k, v))
    for key in ("sinks", "mask"):
        if kw.get(key) is not None:
            kw[key] = kw[key].to(dev).float().contiguous()
    o, lse = fa.splitkv_attention(qd, kd, vd, workspace=workspace, **kw)
    torch.cuda.synchronize()
    return o.cpu(), lse.cpu()


def _check(B, Hq, Hkv, Tq, Tk, d, seed, ctx, **kw):
    q, k, v = workloads.qkv(seed, B, Hq, Hkv, Tq, Tk, d, BF)
    o, lse = splitkv(q, k, v, **kw)
    eo, el = oracle_attention(q, k, v, **kw)
    compare(o, lse, eo, el, BF, ctx)
    return q, k, v, o, lse


@pytest.mark.parametrize("name", sorted(workloads.DECODE))
def test_splitkv_decode_workloads(name):
    w = workloads.DECODE[name]
    p = w.problem
    _check(p.B, p.Hq, p.Hkv, p.Tq, p.Tk, p.d, w.seeds[0], name, scale=p.sm_scale, q_offset=p.q_offset, causal=True)


@pytest.mark.parametrize("Tk", [1, 2, 127, 128, 129, 383, 385, 1000, 4097, 32768])
def test_splitkv_key_lengths(Tk):
    # 2 KV heads: up to 64 splits, capped at two key tiles each; ragged tails
    _check(1, 8, 2, 1, Tk, 64, 500 + Tk, f"split-KV Tk={Tk}", scale=0.125, q_offset=Tk - 1, causal=True)


@pytest.mark.parametrize("d", [64, 96, 128])
def test_splitkv_head_dims(d):
    _check(2, 16, 8, 1, 9000, d, 510 + d, f"split-KV d={d}", scale=d ** -0.5, q_offset=8999, causal=True)


def test_splitkv_one_split_per_head():
    # B * Hkv = 160 >= the SM count: one CTA per KV head, the merge of one partial
    _check(20, 16, 8, 1, 700, 128, 520, "split-KV S=1", scale=128 ** -0.5, q_offset=699, causal=True)


def test_splitkv_sinks():
    # the sink joins the sum once however many splits the range has
    B, Hq, Hkv, Tk, d = 1, 16, 2, 16384, 128
    z = workloads.sinks(53, Hq)
    _check(B, Hq, Hkv, 1, Tk, d, 52, "split-KV sinks", scale=d ** -0.5, q_offset=Tk - 1, causal=True, sinks=z)
    q, k, _ = workloads.qkv(52, B, Hq, Hkv, 1, Tk, d, BF)
    ones = torch.ones((B, Hkv, Tk, d), dtype=BF)
    o, lse = splitkv(q, k, ones, scale=d ** -0.5, q_offset=Tk - 1, causal=True, sinks=z)
    psink = torch.exp(z.double().view(1, -1, 1) - lse.double())
    assert (o.double() - (1.0 - psink)[..., None]).abs().max().item() <= 8e-3


def test_splitkv_window():
    # a window inside a long range: most splits see no key and give empty partials
    _check(1, 32, 4, 1, 20000, 64, 54, "split-KV window", scale=0.125, q_offset=19999, causal=True, window=1500)


def test_splitkv_multi_token_and_mask():
    _check(2, 32, 4, 4, 5000, 128, 55, "split-KV 4 tokens", scale=128 ** -0.5, q_offset=4996, causal=True)
    B, Hq, Hkv, Tq, Tk = 2, 8, 2, 2, 1500
    g = torch.Generator().manual_seed(56)
    mask = torch.randn((B, Hq, Tq, Tk), generator=g)
    mask[torch.rand((B, Hq, Tq, Tk), generator=g) < 0.3] = -float("inf")
    mask[1, 3, 0, :] = -float("inf")  # a fully masked row: zeros, lse = -inf
    strides = (Hq * Tq * Tk, Tq * Tk, Tk, 1)
    *_, o, lse = _check(B, Hq, Hkv, Tq, Tk, 96, 57, "split-KV mask", scale=0.1, q_offset=Tk - 2, causal=True,
                        mask=mask, mask_strides=strides)
    assert torch.isneginf(lse[1, 3, 0]) and torch.all(o[1, 3, 0] == 0)


def test_splitkv_no_keys_visible():
    z = workloads.sinks(58, 8)
    q, k, v = workloads.qkv(58, 1, 8, 2, 1, 3000, 64, BF)
    o, lse = splitkv(q, k, v, scale=0.125, q_offset=5000, causal=True, window=100)
    assert torch.all(o == 0) and torch.all(torch.isneginf(lse))
    o, lse = splitkv(q, k, v, scale=0.125, q_offset=5000, causal=True, window=100, sinks=z)
    assert torch.all(o == 0)
    assert torch.allclose(lse, z.view(1, 8, 1), rtol=0, atol=1e-6)


def test_splitkv_against_fa_fwd_and_repeatable():
    # The long decode step of the benchmark shapes: within rounding of the
    # cluster split of fa_fwd; two calls in a row on one workspace (the
    # counters cleared by each call) give the same bits.
    B, Hq, Hkv, Tk, d = 1, 16, 8, 32768, 128
    q, k, v = workloads.qkv(59, B, Hq, Hkv, 1, Tk, d, BF)
    kw = dict(scale=d ** -0.5, q_offset=Tk - 1, causal=True)
    ref_o, ref_l = gpu_attention(q, k, v, **kw)
    nbytes = fa.fa_splitkv_workspace_bytes(B, Hq, Hkv, 1, d, fa.FA_DTYPE_BF16)
    assert nbytes > 0
    ws = torch.full((nbytes,), 0xFF, dtype=torch.uint8, device="cuda")  # stale contents must not matter
    o1, l1 = splitkv(q, k, v, workspace=ws, **kw)
    o2, l2 = splitkv(q, k, v, workspace=ws, **kw)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert (o1.float() - ref_o.float()).abs().max().item() <= 1e-2
    assert (l1 - ref_l).abs().max().item() <= 1e-3
    eo, el = oracle_attention(q, k, v, **kw)
    compare(o1, l1, eo, el, BF, "split-KV Tk=32768")


def test_splitkv_large_group_is_fa_fwd():
    # group * Tq > 128: not a packed-row call, so the workspace is not used
    # and the result is fa_fwd's bit for bit.
    q, k, v = workloads.qkv(60, 1, 8, 2, 100, 700, 64, BF)
    kw = dict(scale=0.125, q_offset=600, causal=True)
    assert fa.fa_splitkv_workspace_bytes(1, 8, 2, 100, 64, fa.FA_DTYPE_BF16) == 0
    o, lse = splitkv(q, k, v, **kw)
    ref_o, ref_l = gpu_attention(q, k, v, **kw)
    assert torch.equal(o, ref_o) and torch.equal(lse, ref_l)


def test_splitkv_rejects_a_short_workspace():
    q, k, v = (x.cuda() for x in workloads.qkv(61, 1, 8, 2, 1, 4096, 64, BF))
    nbytes = fa.fa_splitkv_workspace_bytes(1, 8, 2, 1, 64, fa.FA_DTYPE_BF16)
    o = torch.zeros((1, 8, 1, 64), dtype=BF, device="cuda")
    lse = torch.zeros((1, 8, 1), dtype=torch.float32, device="cuda")
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    for ptr, size in ((ws, nbytes - 1), (None, nbytes)):
        with pytest.raises(fa.FaError, match="FA_EINVAL"):
            fa.fa_fwd_splitkv(q, k, v, o, lse, 1, 8, 2, 1, 4096, 64, 0.125, 4095, True, 0, None, None, 0, 0, 0, 0,
                              ptr, size, fa.FA_DTYPE_BF16)
    torch.cuda.synchronize()
    assert torch.all(o == 0) and torch.all(lse == 0)  # nothing was launched
