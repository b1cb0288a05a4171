"""GPU parity on long key walks of the tcgen05 kernel.

Units that walk 4096 keys or more take their K and V tiles through many
laps of the rings, so stage and barrier phases wrap many times within one
unit.  The cases combine that with the features that change a unit's key
range (q_offset chunks, no causal rule, a long window with sinks, ragged
query and key tails), checked against the float64 oracle; one check holds
rows of a long causal call bit for bit to the same rows computed by a chunk
call ("FlashAttention forward in C", section 2.4: absolute key tiles make a
row's arithmetic independent of the call it is in).
"""
import numpy as np
import pytest
import torch

import workloads
from parity import compare, compare_fp8, gpu_attention, oracle_attention

pytestmark = pytest.mark.gpu

F8 = torch.float8_e4m3fn


def _inputs(seed, B, Hq, Hkv, Tq, Tk, d, dtype):
    return workloads.qkv(seed, B, Hq, Hkv, Tq, Tk, d, dtype)


def _check(q, k, v, dtype, ctx, **kw):
    o, lse = gpu_attention(q, k, v, **kw)
    eo, el = oracle_attention(q, k, v, **kw)
    if dtype == F8:
        compare_fp8(o, lse, eo, el, v, q.shape[1] // k.shape[1], ctx)
    else:
        compare(o, lse, eo, el, dtype, ctx)


CASES = [
    # (name, B, Hq, Hkv, Tq, Tk, d, q_offset, causal, window, sinks)
    ("causal chunk deep in 4200 keys", 1, 4, 2, 300, 4200, 128, 3900, True, 0, False),
    ("non-causal, 4500 keys, d 64", 2, 4, 2, 200, 4500, 64, 0, False, 0, False),
    ("window 4000 with sinks", 1, 4, 2, 257, 5000, 128, 4743, True, 4000, True),
    ("GQA 4, ragged tails", 1, 8, 2, 130, 4133, 96, 4003, True, 0, False),
]


@pytest.mark.parametrize("dt", ["bf16", "e4m3"])
@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_long_walk(case, dt):
    name, B, Hq, Hkv, Tq, Tk, d, q_offset, causal, window, use_sinks = case
    if dt == "e4m3" and d % 16 != 0:
        pytest.skip("e4m3 rows are whole 16-byte units")
    dtype = torch.bfloat16 if dt == "bf16" else F8
    q, k, v = _inputs(11, B, Hq, Hkv, Tq, Tk, d, dtype)
    z = workloads.sinks(12, Hq) if use_sinks else None
    _check(q, k, v, dtype, f"{name} {dt}", scale=d ** -0.5, q_offset=q_offset, causal=causal, window=window,
           sinks=z)


@pytest.mark.parametrize("dt", ["bf16", "e4m3"])
def test_long_call_and_chunk_rows_agree(dt):
    # One causal call over 4200 positions and the chunk of rows 3000..3299
    # with the keys so far (3300) give the same bits.
    dtype = torch.bfloat16 if dt == "bf16" else F8
    B, Hq, Hkv, T, d = 1, 4, 2, 4200, 128
    q, k, v = _inputs(13, B, Hq, Hkv, T, T, d, dtype)
    o1, l1 = gpu_attention(q, k, v, scale=d ** -0.5, causal=True)
    s, n = 3000, 300
    o2, l2 = gpu_attention(q[:, :, s:s + n].contiguous(), k[:, :, :s + n].contiguous(),
                           v[:, :, :s + n].contiguous(), scale=d ** -0.5, q_offset=s, causal=True)
    assert torch.equal(o1[:, :, s:s + n], o2), "o differs between the long call and the chunk call"
    assert torch.equal(l1[:, :, s:s + n], l2), "lse differs between the long call and the chunk call"
    rows = np.arange(s, s + n, 3, dtype=np.int64)
    eo, el = oracle_attention(q, k, v, rows=rows, scale=d ** -0.5, causal=True)
    if dtype == F8:
        compare_fp8(o1[:, :, rows], l1[:, :, rows], eo, el, v, Hq // Hkv, "4200 causal e4m3")
    else:
        compare(o1[:, :, rows], l1[:, :, rows], eo, el, dtype, "4200 causal bf16")
