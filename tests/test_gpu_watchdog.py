"""Failure detection on the GPU without a fault: every wait in the tensor-core
kernels is bounded.  A test hook makes CTA 0 skip one load, so a wait runs
out; the kernel abandons its work, drains its copies and MMAs, frees tensor
memory and sets its status word.  fa_device_status reports FA_ETIMEOUT, and
the next call on the same context is correct again.
"""
import time

import pytest
import torch

import exact_tiled_attention_flashattention_gb300 as fa
import workloads
from parity import compare, compare_fp8, oracle_attention

pytestmark = pytest.mark.gpu

CASES = [
    # (name, dtype, Hq, Hkv, Tq, Tk, q_offset, fp32_tc)
    ("bf16 prefill", torch.bfloat16, 2, 1, 300, 300, 0, False),
    # walks of up to 35 key tiles: the K and V rings wrap many times per unit
    ("bf16 prefill, long walk", torch.bfloat16, 2, 1, 300, 4396, 4096, False),
    ("e4m3 prefill", torch.float8_e4m3fn, 2, 1, 300, 300, 0, False),
    ("bf16 decode, split key range", torch.bfloat16, 8, 2, 1, 4096, 4095, False),
    ("fp32 on the tensor cores", torch.float32, 2, 1, 300, 300, 0, True),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_wait_runs_out_and_context_survives(case):
    name, dt, Hq, Hkv, Tq, Tk, q_offset, tc = case
    dev = torch.device("cuda", 0)
    q, k, v = workloads.qkv(3, 1, Hq, Hkv, Tq, Tk, 64, dt)
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    kw = dict(scale=0.125, causal=True, q_offset=q_offset, fp32_tc=tc)
    fa.attention(qd, kd, vd, **kw)
    assert fa.fa_device_status() == fa.FA_OK

    fa.fa_test_drop_arrive(True)
    try:
        t0 = time.time()
        fa.attention(qd, kd, vd, **kw)
        st = fa.fa_device_status(check=False)
        msg = fa.fa_last_error()  # before the next fa_* call resets it
        took = time.time() - t0
    finally:
        fa.fa_test_drop_arrive(False)
    assert st == fa.FA_ETIMEOUT, (name, st, msg)
    assert "bounded wait" in msg
    assert took < 30.0, took  # two-second waits, then bounded drains
    assert fa.fa_device_status() == fa.FA_OK  # the word was cleared

    o, lse = fa.attention(qd, kd, vd, **kw)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == fa.FA_OK
    eo, el = oracle_attention(q, k, v, scale=0.125, causal=True, q_offset=q_offset)
    if dt == torch.float8_e4m3fn:
        compare_fp8(o.cpu(), lse.cpu(), eo, el, v, Hq // Hkv, f"{name}: after the timeout")
    else:
        compare(o.cpu(), lse.cpu(), eo, el, dt, f"{name}: after the timeout")
