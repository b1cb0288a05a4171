"""Variable-length batches (fa_fwd_varlen): sequences packed along the rows of
[total, H, d] tensors with cu_seqlens offsets.  Each sequence must equal a
call on that sequence alone, bit for bit, and the oracle within tolerance."""
import numpy as np
import pytest
import torch

import exact_tiled_attention_flashattention_gb300 as fa
import workloads
from parity import compare, compare_fp8, oracle_attention

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "bf16": torch.bfloat16, "e4m3": torch.float8_e4m3fn}
DEV = torch.device("cuda", 0)


def _pack(ts):
    """[1, H, T_i, d] tensors -> [sum T_i, H, d] and the cu_seqlens table."""
    cu = [0]
    for t in ts:
        cu.append(cu[-1] + t.shape[2])
    packed = torch.cat([t[0].transpose(0, 1) for t in ts], dim=0)  # [T, H, d]
    return packed, torch.tensor(cu, dtype=torch.int32)


def _run(dt, lens_q, lens_k, Hq, Hkv, d, seed, **kw):
    qs, ks, vs = [], [], []
    for i, (tq, tk) in enumerate(zip(lens_q, lens_k)):
        q, k, v = workloads.qkv(seed + i, 1, Hq, Hkv, tq, tk, d, DT[dt])
        qs.append(q), ks.append(k), vs.append(v)
    qp, cuq = _pack(qs)
    kp, cuk = _pack(ks)
    vp, _ = _pack(vs)
    o, lse = fa.varlen_attention(qp.to(DEV), kp.to(DEV), vp.to(DEV), cuq.to(DEV), cuk.to(DEV), max(lens_q),
                                 max(lens_k), **kw)
    torch.cuda.synchronize()
    o, lse = o.cpu(), lse.cpu()
    for i, (tq, tk) in enumerate(zip(lens_q, lens_k)):
        a, b = int(cuq[i]), int(cuq[i + 1])
        oi = o[a:b].transpose(0, 1).unsqueeze(0)  # [1, Hq, tq, d]
        li = lse[:, a:b].unsqueeze(0)
        if tq == 0:
            continue
        # the same sequence alone: its queries are its last positions (positions
        # do not matter without a causal rule or a window)
        off = tk - tq if (kw.get("causal", True) or kw.get("window", 0)) else 0
        o1, l1 = fa.attention(qs[i].to(DEV), ks[i].to(DEV), vs[i].to(DEV), q_offset=off, **kw)
        torch.cuda.synchronize()
        assert torch.equal(oi, o1.cpu()) and torch.equal(li, l1.cpu()), f"sequence {i}"
        eo, el = oracle_attention(qs[i], ks[i], vs[i], q_offset=off, **kw)
        if dt == "e4m3":
            compare_fp8(oi, li, eo, el, vs[i], Hq // Hkv, f"varlen {dt} seq {i} ({tq}x{tk})")
        else:
            compare(oi, li, eo, el, DT[dt], f"varlen {dt} seq {i} ({tq}x{tk})")


@pytest.mark.parametrize("dt", ["bf16", "f32", "e4m3"])
def test_varlen_causal_prefill(dt):
    lens = [1, 100, 511, 129, 1000]
    _run(dt, lens, lens, 8, 4, 64, 90, scale=0.125, causal=True)


@pytest.mark.parametrize("dt", ["bf16", "f32", "e4m3"])
def test_varlen_chunks_and_empty(dt):
    # queries as the last positions of longer key ranges; one empty sequence
    lq = [200, 0, 37, 300]
    lk = [700, 50, 37, 2100]
    _run(dt, lq, lk, 12, 4, 128, 91, scale=128 ** -0.5, causal=True)


@pytest.mark.parametrize("dt", ["bf16", "e4m3"])
def test_varlen_window_sinks(dt):
    lens = [400, 260, 1500]
    z = workloads.sinks(93, 6).to(DEV)
    _run(dt, lens, lens, 6, 2, 96, 92, scale=0.1, causal=True, window=150, sinks=z)


def test_varlen_noncausal_f32():
    _run("f32", [70, 300], [90, 200], 4, 4, 64, 94, scale=0.125, causal=False)
