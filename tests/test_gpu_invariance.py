"""GPU-vs-GPU bitwise properties ("FlashAttention forward in C", section 2.4
and its test catalogue): a row's bits do not depend on chunking through
q_offset, on the batch it sits in, or on the run.  Every dtype: fp32 on the
SIMT and on the tensor-core path, bf16 and e4m3.
"""
import pytest
import torch

import workloads
from parity import gpu_attention

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "f32tc": torch.float32, "bf16": torch.bfloat16, "e4m3": torch.float8_e4m3fn}
ALL = ["f32", "f32tc", "bf16", "e4m3"]


def _run(dt, *args, **kw):
    return gpu_attention(*args, fp32_tc=(dt == "f32tc"), **kw)


@pytest.mark.parametrize("dt", ALL)
@pytest.mark.parametrize("chunk", [1, 3, 5, 16, 100])
def test_chunk_invariance(dt, chunk):
    T = 300
    q, k, v = workloads.qkv(21, 1, 4, 2, T, T, 64, DT[dt])
    o1, l1 = _run(dt, q, k, v, scale=0.125, causal=True, window=70)
    outs, lses = [], []
    for start, n in workloads.chunk_ranges(T, chunk):
        o, l = _run(dt, q[:, :, start:start + n].contiguous(), k[:, :, :start + n].contiguous(),
                             v[:, :, :start + n].contiguous(), scale=0.125, q_offset=start, causal=True, window=70)
        outs.append(o)
        lses.append(l)
    assert torch.equal(torch.cat(outs, 2), o1)
    assert torch.equal(torch.cat(lses, 2), l1)


@pytest.mark.parametrize("dt", ALL)
def test_batch_invariance(dt):
    q, k, v = workloads.qkv(22, 3, 4, 2, 200, 200, 64, DT[dt])
    ob, lb = _run(dt, q, k, v, scale=0.125, causal=True)
    for b in range(3):
        o, l = _run(dt, q[b:b + 1].contiguous(), k[b:b + 1].contiguous(), v[b:b + 1].contiguous(), scale=0.125,
                             causal=True)
        assert torch.equal(o, ob[b:b + 1]) and torch.equal(l, lb[b:b + 1])


@pytest.mark.parametrize("dt", ALL)
def test_run_to_run(dt):
    q, k, v = workloads.qkv(23, 1, 16, 8, 1000, 1000, 128, DT[dt])
    a = _run(dt, q, k, v, scale=128 ** -0.5, causal=True)
    b = _run(dt, q, k, v, scale=128 ** -0.5, causal=True)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
