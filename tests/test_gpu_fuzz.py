"""Seeded random shapes and flags on every dtype, against the float64 oracle.

Each case draws batch, heads (GQA group 1-4), query and key lengths (with
ragged tails, Tk = 0, single rows), d within the dtype's range, the causal
rule, q_offset, a window, sinks and an additive mask (broadcast or full, with
-inf entries and some fully masked rows) from a fixed seed, runs the CUDA
path and compares it with the oracle at the dtype's tolerance: fp32 (SIMT
and tensor cores) 1e-4, bf16 2e-2 / 2e-3 / 1e-2, e4m3 the per-element bound
of its P and O rounding.  The cases are small enough for the oracle to
finish in seconds; together they reach combinations the hand-picked cases do
not.
"""
import math

import numpy as np
import pytest
import torch

import workloads
from parity import compare, compare_fp8, gpu_attention, oracle_attention

pytestmark = pytest.mark.gpu

F8 = torch.float8_e4m3fn
DTYPES = ("f32", "f32tc", "bf16", "e4m3")
# d values each path accepts: fp32 even up to 256, TF32 multiples of 4 up to
# 128, bf16 multiples of 8 up to 128, e4m3 multiples of 16 up to 128.
D_CHOICES = {"f32": [2, 6, 32, 64, 100, 128, 160, 256], "f32tc": [4, 12, 36, 64, 96, 128],
             "bf16": [8, 24, 64, 72, 96, 128], "e4m3": [16, 32, 48, 64, 112, 128]}
CASES_PER_DTYPE = 30


def _draw(rng, dt):
    """One random case: sizes, flags and the seeds of its inputs."""
    group = int(rng.choice([1, 1, 2, 3, 4]))
    Hkv = int(rng.integers(1, 4))
    c = dict(B=int(rng.integers(1, 4)), Hkv=Hkv, Hq=Hkv * group, d=int(rng.choice(D_CHOICES[dt])))
    c["Tq"] = int(rng.choice([1, 2, 7, 63, 64, 65, 127, 129, 200, 257, 300]))
    c["causal"] = bool(rng.random() < 0.7)
    c["q_offset"] = int(rng.choice([0, 0, 1, 5, 100, 250]))
    extra = int(rng.choice([0, 0, 1, 17, 128, 133]))
    c["Tk"] = max(0, c["q_offset"] + c["Tq"] + extra - (int(rng.integers(0, 40)) if rng.random() < 0.3 else 0))
    if rng.random() < 0.05:
        c["Tk"] = 0
    c["window"] = int(rng.choice([0, 0, 0, 1, 16, 128, 200]))
    c["sinks"] = bool(rng.random() < 0.3)
    c["mask"] = str(rng.choice(["none", "none", "none", "broadcast", "full"]))
    c["seed"] = int(rng.integers(0, 1 << 30))
    return c


def _cases():
    rng = np.random.default_rng(20261202)
    out = []
    for dt in DTYPES:
        for n in range(CASES_PER_DTYPE):
            out.append((dt, n, _draw(rng, dt)))
    return out


CASES = _cases()


@pytest.mark.parametrize("dt,n,c", CASES, ids=[f"{dt}-{n}" for dt, n, _ in CASES])
def test_fuzz(dt, n, c):
    tdt = {"f32": torch.float32, "f32tc": torch.float32, "bf16": torch.bfloat16, "e4m3": F8}[dt]
    B, Hq, Hkv, Tq, Tk, d = c["B"], c["Hq"], c["Hkv"], c["Tq"], c["Tk"], c["d"]
    q, k, v = workloads.qkv(c["seed"], B, Hq, Hkv, Tq, Tk, d, tdt)
    z = workloads.sinks(c["seed"] + 1, Hq) if c["sinks"] else None
    mask, strides = None, (0, 0, 0, 0)
    if c["mask"] != "none" and Tk > 0:
        g = torch.Generator().manual_seed(c["seed"] + 2)
        if c["mask"] == "broadcast":  # one [Tq, Tk] mask for every batch and head
            mask = torch.randn((Tq, Tk), generator=g)
            strides = (0, 0, Tk, 1)
        else:
            mask = torch.randn((B, Hq, Tq, Tk), generator=g)
            strides = (Hq * Tq * Tk, Tq * Tk, Tk, 1)
        mask[torch.rand(mask.shape, generator=g) < 0.15] = -math.inf
        mask.view(-1, Tk)[:: 7] = -math.inf  # every 7th row sees no key
    kw = dict(scale=1.0 / math.sqrt(d), q_offset=c["q_offset"], causal=c["causal"], window=c["window"], sinks=z,
              mask=mask, mask_strides=strides)
    o, lse = gpu_attention(q, k, v, fp32_tc=(dt == "f32tc"), **kw)
    eo, el = oracle_attention(q, k, v, **kw)
    ctx = f"{dt} case {n} {c}"
    if dt == "e4m3":
        compare_fp8(o, lse, eo, el, v, Hq // Hkv, ctx)
    else:
        compare(o, lse, eo, el, tdt, ctx)
