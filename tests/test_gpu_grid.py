"""Grid-size invariance of the persistent tensor-core kernels.

"FlashAttention forward in C", section 4 (its test catalogue) holds the
thread-pool result to the serial one bit for bit
(pool_result_equals_serial_bitwise): the workers never change a row's bits.
On the GPU the workers are the CTAs of a persistent grid, which hand out units
by grid size and carry ring, S-buffer and barrier state from one unit to the
next.  fa_test_max_ctas caps the grid; a row's output and lse must be the same
with one CTA walking every unit, with a few CTAs, and with one CTA per SM.

The fp32 tensor-core kernel launches one CTA per query tile (its grid is fixed
by the problem, not by the SM count), so the cap does not reach it; its runs
are compared anyway, as a run-to-run check of that path.
"""
import pytest
import torch

import exact_tiled_attention_flashattention_gb300 as fa
import workloads

pytestmark = pytest.mark.gpu

DT = {"bf16": torch.bfloat16, "e4m3": torch.float8_e4m3fn, "f32tc": torch.float32}


def _attention_capped(cap, q, k, v, **kw):
    fa.fa_test_max_ctas(cap)
    try:
        o, lse = fa.attention(q, k, v, **kw)
        torch.cuda.synchronize()
    finally:
        fa.fa_test_max_ctas(0)
    return o, lse


@pytest.mark.parametrize("dt", ["bf16", "e4m3", "f32tc"])
def test_long_prefill_grid_sizes(dt):
    """T = 2044, 16 query heads on 8 KV heads, d = 128, causal: 256 units of
    1 to 16 key tiles; grids of 1, 7 and (0) one CTA per SM."""
    T = 2044
    q, k, v = workloads.qkv(100, 1, 16, 8, T, T, 128, DT[dt])
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    kw = dict(scale=128 ** -0.5, causal=True, fp32_tc=(dt == "f32tc"))
    ref_o, ref_l = _attention_capped(0, q, k, v, **kw)
    for cap in (1, 7):
        o, lse = _attention_capped(cap, q, k, v, **kw)
        assert torch.equal(o, ref_o), f"{dt}: output differs with the grid capped at {cap}"
        assert torch.equal(lse, ref_l), f"{dt}: lse differs with the grid capped at {cap}"


@pytest.mark.parametrize("dt", ["bf16", "e4m3"])
def test_window_sinks_grid_sizes(dt):
    """A window with sinks, q_offset and a ragged tail: units whose walks
    start past key 0 and end on a partial tile; grids of 1, 3, 5 and full."""
    T, Tq = 900, 700
    q, k, v = workloads.qkv(31, 2, 8, 2, Tq, T, 64, DT[dt])
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    sinks = torch.randn(8, generator=torch.Generator().manual_seed(5)).cuda()
    kw = dict(scale=0.125, q_offset=T - Tq, causal=True, window=200, sinks=sinks)
    ref_o, ref_l = _attention_capped(0, q, k, v, **kw)
    for cap in (1, 3, 5):
        o, lse = _attention_capped(cap, q, k, v, **kw)
        assert torch.equal(o, ref_o) and torch.equal(lse, ref_l), f"{dt}: grid capped at {cap}"


def test_varlen_grid_sizes():
    """Variable-length batch (the persistent row mapping with per-sequence
    lengths): grids of 1, 2 and full."""
    lens = [130, 517, 64, 1000]
    H, Hkv, d = 4, 2, 128
    total = sum(lens)
    q, k, v = workloads.qkv(41, 1, H, Hkv, total, total, d, torch.bfloat16)
    # [1, H, total, d] -> [total, H, d]: the sequences packed along the rows
    q, k, v = (x[0].transpose(0, 1).contiguous().cuda() for x in (q, k, v))
    cu = torch.tensor([0] + list(torch.tensor(lens).cumsum(0)), dtype=torch.int32).cuda()

    def run(cap):
        fa.fa_test_max_ctas(cap)
        try:
            o, lse = fa.varlen_attention(q, k, v, cu, cu, max(lens), max(lens), scale=d ** -0.5, causal=True)
            torch.cuda.synchronize()
        finally:
            fa.fa_test_max_ctas(0)
        return o, lse

    ref = run(0)
    for cap in (1, 2):
        got = run(cap)
        assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1]), f"grid capped at {cap}"
