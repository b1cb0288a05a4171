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


def sample_rows(T):
    """First 256, last 256 and every 127th row (deterministic)."""
    rows = set(range(min(256, T))) | set(range(max(0, T - 256), T)) | set(range(0, T, 127))
    return np.array(sorted(rows), dtype=np.int64)
