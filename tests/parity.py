"""Helpers for the GPU parity tests: run the CUDA path through the C ABI,
run the float64 oracle on the same (rounded) inputs, compare within the
stated tolerances.

Tolerances (fixed by the method's statement of the target):
  fp32: max |o - oracle| <= 1e-4 and max |lse - oracle| <= 1e-4;
  bf16 (oracle on the same bf16-rounded inputs): max |o - oracle| <= 2e-2,
        mean |o - oracle| <= 2e-3, max |lse - oracle| <= 1e-2.
Rows the oracle calls empty (lse = -inf) must have lse = -inf and o exactly 0
on the GPU.
"""
from __future__ import annotations

import numpy as np
import torch

import exact_tiled_attention_flashattention_gb300 as fa
import oracle

TOL = {
    torch.float32: dict(o_max=1e-4, o_mean=1e-4, lse_max=1e-4),
    torch.bfloat16: dict(o_max=2e-2, o_mean=2e-3, lse_max=1e-2),
}


def gpu_attention(q, k, v, *, scale, q_offset=0, causal=True, window=0, sinks=None, mask=None,
                  mask_strides=(0, 0, 0, 0), fp32_tc=False):
    """CUDA path through fa_fwd; CPU tensors in, CPU tensors out.  ``fp32_tc``
    selects the three-TF32 tensor-core path for fp32 inputs."""
    dev = torch.device("cuda", 0)
    qd, kd, vd = q.to(dev).contiguous(), k.to(dev).contiguous(), v.to(dev).contiguous()
    sd = sinks.to(dev).float().contiguous() if sinks is not None else None
    md = mask.to(dev).float().contiguous() if mask is not None else None
    o, lse = fa.attention(qd, kd, vd, scale=scale, q_offset=q_offset, causal=causal, window=window, sinks=sd,
                          mask=md, mask_strides=mask_strides, fp32_tc=fp32_tc)
    torch.cuda.synchronize()
    return o.cpu(), lse.cpu()


def oracle_attention(q, k, v, *, scale, q_offset=0, causal=True, window=0, sinks=None, mask=None,
                     mask_strides=(0, 0, 0, 0), rows=None):
    f = lambda t: None if t is None else t.detach().cpu().float().numpy()  # exact widening of fp32 / bf16
    return oracle.attention(f(q), f(k), f(v), scale, q_offset=q_offset, causal=causal, window=window,
                            sinks=f(sinks), mask=None if mask is None else f(mask).reshape(-1),
                            mask_strides=mask_strides, rows=rows)


def compare(o, lse, eo, el, dtype, ctx=""):
    """Assert the GPU result (o, lse: torch CPU) matches the oracle (eo, el)."""
    tol = TOL[dtype]
    o = o.float().numpy().astype(np.float64)
    lse = lse.numpy().astype(np.float64)
    empty = np.isneginf(el)
    assert np.array_equal(np.isneginf(lse), empty), f"{ctx}: empty-row pattern differs"
    assert np.all(o[empty] == 0.0), f"{ctx}: empty rows must give o = 0"
    assert np.all(np.isfinite(lse[~empty])), f"{ctx}: non-finite lse on a non-empty row"
    d_o = np.abs(o - eo)
    d_l = np.abs(lse[~empty] - el[~empty]) if (~empty).any() else np.zeros(1)
    msg = (f"{ctx}: max|do|={d_o.max():.3g} mean|do|={d_o.mean():.3g} max|dlse|={d_l.max():.3g} "
           f"(tol {tol})")
    assert np.all(np.isfinite(o)), msg
    assert d_o.max() <= tol["o_max"], msg
    assert d_o.mean() <= tol["o_mean"], msg
    assert d_l.max() <= tol["lse_max"], msg
    return d_o.max(), d_o.mean(), d_l.max()


# e4m3 inputs (the oracle sees the same e4m3 values, widened exactly).  The
# kernel rounds P to e4m3 (3 mantissa bits: each weight off by at most 2^-4
# of itself) and O to bf16 (2^-9), and l sums the unrounded p, so per element
#     |o - o_ref| <= 2^-4 max_j |v_j[x]| + 2^-8 |o_ref|
# whatever the shape.  On the causal prefill workloads (T = 511 and 2044) a
# float64 simulation of exactly this arithmetic gives max 2.7e-2 and mean
# 2.2e-3 on O; those checks take twice the max, and every workload check takes
# twice the mean.  S = Q K^T is exact products summed in fp32 and lse uses
# only fp32 arithmetic: 1e-4, the fp32 bound.
FP8_TOL = dict(o_max=6e-2, o_mean=5e-3, lse_max=1e-4)


def compare_fp8(o, lse, eo, el, v, group, ctx="", workload=False, causal_prefill=False):
    """GPU result (o bf16, lse: torch CPU) against the oracle for e4m3 inputs.
    v: the e4m3 values [B, Hkv, Tk, d] (CPU); group = Hq / Hkv.  `workload`
    adds the mean limit, `causal_prefill` the simulated max as well."""
    o = o.float().numpy().astype(np.float64)
    lse = lse.numpy().astype(np.float64)
    empty = np.isneginf(el)
    assert np.array_equal(np.isneginf(lse), empty), f"{ctx}: empty-row pattern differs"
    assert np.all(o[empty] == 0.0), f"{ctx}: empty rows must give o = 0"
    assert np.all(np.isfinite(o)), f"{ctx}: non-finite o"
    vf = v.float().numpy().astype(np.float64)
    vmax = np.abs(vf).max(axis=2) if vf.shape[2] > 0 else np.zeros(vf.shape[:2] + vf.shape[3:])
    vmax = np.repeat(vmax, group, axis=1)[:, :, None, :]  # [B, Hq, 1, d]
    d_o = np.abs(o - eo)
    bound = 2.0 ** -4 * vmax + 2.0 ** -8 * np.abs(eo) + 1e-6
    worst = (d_o - bound).max() if d_o.size else 0.0
    d_l = np.abs(lse[~empty] - el[~empty]) if (~empty).any() else np.zeros(1)
    msg = f"{ctx}: max|do|={d_o.max():.3g} mean|do|={d_o.mean():.3g} max|dlse|={d_l.max():.3g}"
    assert worst <= 0.0, f"{msg}: over the per-element bound by {worst:.3g}"
    assert d_l.max() <= FP8_TOL["lse_max"], msg
    if workload or causal_prefill:
        assert d_o.mean() <= FP8_TOL["o_mean"], msg
    if causal_prefill:
        assert d_o.max() <= FP8_TOL["o_max"], msg
    return d_o.max(), d_o.mean(), d_l.max()


def sample_rows(T):
    """First 256, last 256 and every 127th row (deterministic)."""
    rows = set(range(min(256, T))) | set(range(max(0, T - 256), T)) | set(range(0, T, 127))
    return np.array(sorted(rows), dtype=np.int64)
