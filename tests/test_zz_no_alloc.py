"""The split-KV entry point that allocates nothing (fa_fwd_splitkv_noalloc).

Some callers cannot call cudaMalloc: an engine whose memory planner already
owns the GPU's memory, a plugin whose host forbids allocation while it runs, a
loop where cudaMalloc's possible device synchronisation would stall the
pipeline.  For them the library keeps the split-KV workspace in a static
device array of FA_SPLITKV_NOALLOC_MAX_SCRATCH bytes.  That array is shared
by every call on a GPU and keeps the previous call's contents.

The test calls the entry point through the C ABI twice in a row, on two
different decode problems, so that the second call starts from the first
one's leftovers.  It checks each output against fa_fwd_splitkv with a
workspace of its own, within the bf16 tolerances of the parity tests.  A call
whose workspace would exceed the array must be refused, with nothing
launched.  The file runs last, and it passes both alone and after the rest of
the suite: the array's first use on the device may come from this file or
from an earlier one.
"""
import numpy as np
import pytest
import torch

import exact_tiled_attention_flashattention_gb300 as fa
import workloads
from parity import TOL

pytestmark = pytest.mark.gpu

BF = torch.bfloat16


def _problem(seed, B, Hq, Hkv, Tq, Tk, d, with_sinks):
    q, k, v = (x.cuda() for x in workloads.qkv(seed, B, Hq, Hkv, Tq, Tk, d, BF))
    sinks = workloads.sinks(seed + 1, Hq).cuda() if with_sinks else None
    return dict(q=q, k=k, v=v, sinks=sinks, B=B, Hq=Hq, Hkv=Hkv, Tq=Tq, Tk=Tk, d=d, scale=d ** -0.5,
                q_offset=Tk - Tq)


def _outputs(p):
    o = torch.full((p["B"], p["Hq"], p["Tq"], p["d"]), float("nan"), dtype=BF, device="cuda")
    lse = torch.full((p["B"], p["Hq"], p["Tq"]), float("nan"), dtype=torch.float32, device="cuda")
    return o, lse


def _args(p, o, lse):
    return (p["q"], p["k"], p["v"], o, lse, p["B"], p["Hq"], p["Hkv"], p["Tq"], p["Tk"], p["d"], p["scale"],
            p["q_offset"], True, 0, p["sinks"], None, 0, 0, 0, 0)


def _with_workspace(p):
    """The same call through fa_fwd_splitkv, with a workspace allocated here."""
    o, lse = _outputs(p)
    n = fa.fa_splitkv_workspace_bytes(p["B"], p["Hq"], p["Hkv"], p["Tq"], p["d"], fa.FA_DTYPE_BF16)
    ws = torch.empty(max(n, 1), dtype=torch.uint8, device="cuda")
    fa.fa_fwd_splitkv(*_args(p, o, lse), ws, n, fa.FA_DTYPE_BF16)
    torch.cuda.synchronize()
    return o.cpu(), lse.cpu()


def _within_tolerance(o, lse, ref_o, ref_l, ctx):
    tol = TOL[BF]
    o, ref_o = o.double().numpy(), ref_o.double().numpy()
    lse, ref_l = lse.double().numpy(), ref_l.double().numpy()
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse)), f"{ctx}: an output was not written"
    d_o = np.abs(o - ref_o)
    assert d_o.max() <= tol["o_max"] and d_o.mean() <= tol["o_mean"], f"{ctx}: max|do|={d_o.max():.3g}"
    assert np.abs(lse - ref_l).max() <= tol["lse_max"], f"{ctx}: lse"


def test_no_alloc_matches_the_workspace_entry_point_on_two_calls_in_a_row():
    first = _problem(900, 1, 16, 8, 1, 32768, 128, with_sinks=False)  # 8 KV heads over every SM
    second = _problem(910, 2, 32, 4, 2, 5000, 64, with_sinks=True)    # other sizes, a sink per head
    for p in (first, second):
        need = fa.fa_splitkv_workspace_bytes(p["B"], p["Hq"], p["Hkv"], p["Tq"], p["d"], fa.FA_DTYPE_BF16)
        assert 0 < need <= fa.FA_SPLITKV_NOALLOC_MAX_SCRATCH
    o1, l1 = _outputs(first)
    o2, l2 = _outputs(second)
    # Two calls in a row on one stream: the second finds the first's counters
    # and partials in the shared array.
    fa.fa_fwd_splitkv_noalloc(*_args(first, o1, l1), fa.FA_DTYPE_BF16)
    fa.fa_fwd_splitkv_noalloc(*_args(second, o2, l2), fa.FA_DTYPE_BF16)
    torch.cuda.synchronize()
    _within_tolerance(o1.cpu(), l1.cpu(), *_with_workspace(first), "first call")
    _within_tolerance(o2.cpu(), l2.cpu(), *_with_workspace(second), "second call")


def test_no_alloc_refuses_a_call_beyond_its_array():
    # 160 KV heads with 128 packed rows each need about 10 MiB of partials.
    p = _problem(920, 20, 128, 8, 8, 256, 128, with_sinks=False)
    need = fa.fa_splitkv_workspace_bytes(p["B"], p["Hq"], p["Hkv"], p["Tq"], p["d"], fa.FA_DTYPE_BF16)
    assert need > fa.FA_SPLITKV_NOALLOC_MAX_SCRATCH
    o, lse = _outputs(p)
    with pytest.raises(fa.FaError, match="FA_EUNSUPPORTED.*scratch"):
        fa.fa_fwd_splitkv_noalloc(*_args(p, o, lse), fa.FA_DTYPE_BF16)
    torch.cuda.synchronize()
    assert torch.isnan(o.float()).all() and torch.isnan(lse).all()  # nothing was launched
