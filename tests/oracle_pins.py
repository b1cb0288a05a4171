"""Pins of the float64 oracle against facts fixed outside it.

Each pin takes an ``oracle.Oracle`` (the real build or a planted mutant) and
raises AssertionError when the oracle disagrees with:
  * values printed on the pages (the worked example, "FlashAttention forward
    in C", section 3, stored under tests/golden/ with its citation);
  * identities the pages state (the sink identity and the empty-row contract
    of the same page's test catalogue, section 4; weights summing to 1);
  * closed forms (a single key, a window of one, a zero query, a constant
    shift of the logits);
  * a float64 library routine (torch's scaled_dot_product_attention and
    logsumexp) on tiny shapes, with the visible key set enumerated as index
    ranges by brute force and the sink emulated as one extra zero key.

The pins are kept free of the oracle's own code: none of them calls into it
except through its public entry point.
"""
from __future__ import annotations

import itertools
import math
from pathlib import Path

import numpy as np
import torch

GOLDEN = Path(__file__).resolve().parent / "golden"


def _read_golden(name):
    vals = {}
    for line in (GOLDEN / name).read_text().splitlines():
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, rhs = line.split("=", 1)
        vals[key.strip()] = np.array([float(x) for x in rhs.split()], dtype=np.float64)
    return vals


def _rng(seed):
    return np.random.default_rng(seed)


# ----------------------------------------------------------------------------
# Values printed on the pages
# ----------------------------------------------------------------------------

def pin_worked_example(orc):
    g = _read_golden("worked_example.txt")
    q = g["q"].reshape(1, 1, 1, 2)
    k = np.stack([g["k0"], g["k1"], g["k2"]]).reshape(1, 1, 3, 2)
    v = np.stack([g["v0"], g["v1"], g["v2"]]).reshape(1, 1, 3, 2)
    scale = float(g["scale"][0])
    o, lse = orc.attention(q, k, v, scale, causal=False, threads=1)
    # printed "exactly" [3, 4]; lse printed to 7 decimals
    assert np.allclose(o.reshape(2), g["o"], rtol=0, atol=1e-12), o
    assert abs(lse.item() - g["lse"][0]) <= 6e-8, lse
    o2, lse2 = orc.attention(q, k, v, scale, causal=True, q_offset=1, threads=1)
    assert np.allclose(o2.reshape(2), g["causal_q_offset1_o"], rtol=0, atol=6e-8), o2
    # not printed: with keys 0 and 1 only, lse = 1 + ln(1 + e^-1)
    assert abs(lse2.item() - (1.0 + math.log1p(math.exp(-1.0)))) <= 1e-12, lse2


def pin_sink_identity(orc):
    # All-ones values with a sink: weights sum to 1 - p_sink = 2/3 and lse = ln 3
    # (section 4, sinks_join_the_denominator).  Shape reconstructed: q = 0,
    # two visible keys, z = 0, so each of the three logits is 0.
    q = np.zeros((1, 1, 1, 4))
    k = _rng(1).standard_normal((1, 1, 2, 4))
    v = np.ones((1, 1, 2, 4))
    o, lse = orc.attention(q, k, v, 0.5, causal=False, sinks=np.zeros(1), threads=1)
    assert np.allclose(o, 2.0 / 3.0, rtol=0, atol=1e-15), o
    assert abs(lse.item() - math.log(3.0)) <= 1e-15, lse


# ----------------------------------------------------------------------------
# Identities and contracts
# ----------------------------------------------------------------------------

def pin_sink_weights_sum(orc):
    # V == 1 with sinks: every component of o equals 1 - e^{z_h - lse}.
    r = _rng(2)
    B, Hq, Hkv, Tq, Tk, D = 2, 4, 2, 9, 13, 8
    q = r.standard_normal((B, Hq, Tq, D))
    k = r.standard_normal((B, Hkv, Tk, D))
    v = np.ones((B, Hkv, Tk, D))
    z = r.standard_normal(Hq) * 2.0
    for causal, window, qoff in [(True, 0, 4), (True, 3, 4), (False, 5, 7), (False, 0, 0)]:
        o, lse = orc.attention(q, k, v, 0.7, causal=causal, window=window, q_offset=qoff,
                               sinks=z, threads=2)
        psink = np.exp(z[None, :, None] - lse)
        assert np.allclose(o, (1.0 - psink)[..., None], rtol=0, atol=1e-12)


def pin_weights_sum_to_one(orc):
    r = _rng(3)
    B, Hq, Hkv, Tq, Tk, D = 1, 6, 2, 11, 11, 5
    q = r.standard_normal((B, Hq, Tq, D))
    k = r.standard_normal((B, Hkv, Tk, D))
    v = np.ones((B, Hkv, Tk, D))
    o, lse = orc.attention(q, k, v, 0.3, causal=True, window=4, threads=3)
    assert np.all(np.isfinite(lse))
    assert np.allclose(o, 1.0, rtol=0, atol=1e-13)


def pin_empty_rows(orc):
    # A query whose window excludes every key: zeros and -inf; with a sink,
    # zeros and lse = the sink (section 4, no_visible_key_gives_zeros_and_minus_inf).
    r = _rng(4)
    q = r.standard_normal((1, 2, 3, 4))
    k = r.standard_normal((1, 1, 3, 4))
    v = r.standard_normal((1, 1, 3, 4))
    o, lse = orc.attention(q, k, v, 1.0, causal=True, window=2, q_offset=10, threads=1)
    assert np.all(o == 0.0) and np.all(lse == -np.inf), (o, lse)
    z = np.array([0.25, -1.5])
    o, lse = orc.attention(q, k, v, 1.0, causal=True, window=2, q_offset=10, sinks=z, threads=1)
    assert np.all(o == 0.0), o
    assert np.array_equal(lse, np.broadcast_to(z[None, :, None], lse.shape)), lse
    # Tk == 0 gives zeros as well.
    k0 = np.zeros((1, 1, 0, 4))
    o, lse = orc.attention(q, k0, k0, 1.0, causal=False, threads=1)
    assert np.all(o == 0.0) and np.all(lse == -np.inf)
    # A row that the additive mask removes entirely is empty too.
    mask = np.zeros((3, 3))
    mask[1, :] = -np.inf
    o, lse = orc.attention(q, k, v, 1.0, causal=False, mask=mask, mask_strides=(0, 0, 3, 1), threads=1)
    assert np.all(o[:, :, 1] == 0.0) and np.all(lse[:, :, 1] == -np.inf)
    assert np.all(np.isfinite(lse[:, :, [0, 2]]))


def pin_single_key(orc):
    # Tk = 1: o = v_0 and lse = s_0 = scale q.k_0 + mask.
    r = _rng(5)
    q = r.standard_normal((1, 3, 4, 6))
    k = r.standard_normal((1, 3, 1, 6))
    v = r.standard_normal((1, 3, 1, 6))
    mask = r.standard_normal((4, 1))
    o, lse = orc.attention(q, k, v, 0.4, causal=False, mask=mask, mask_strides=(0, 0, 1, 1), threads=1)
    for h in range(3):
        for i in range(4):
            assert np.allclose(o[0, h, i], v[0, h, 0], rtol=0, atol=1e-15)
            s0 = 0.4 * float(np.dot(q[0, h, i], k[0, h, 0])) + mask[i, 0]
            assert abs(lse[0, h, i] - s0) <= 1e-13


def pin_window_one(orc):
    # causal with a window of 1: each row sees exactly its own position.
    r = _rng(6)
    Tq, Tk, off = 5, 9, 3
    q = r.standard_normal((1, 2, Tq, 4))
    k = r.standard_normal((1, 2, Tk, 4))
    v = r.standard_normal((1, 2, Tk, 4))
    o, lse = orc.attention(q, k, v, 0.9, causal=True, window=1, q_offset=off, threads=1)
    for h in range(2):
        for i in range(Tq):
            p = off + i
            assert np.allclose(o[0, h, i], v[0, h, p], rtol=0, atol=1e-15)
            assert abs(lse[0, h, i] - 0.9 * float(np.dot(q[0, h, i], k[0, h, p]))) <= 1e-13


def pin_zero_query_uniform(orc):
    # q = 0: equal weights over the visible keys; o is their mean, lse = ln |V_i|.
    r = _rng(7)
    Tq, Tk, off, w = 6, 12, 4, 5
    q = np.zeros((1, 1, Tq, 3))
    k = r.standard_normal((1, 1, Tk, 3))
    v = r.standard_normal((1, 1, Tk, 3))
    o, lse = orc.attention(q, k, v, 1.0, causal=True, window=w, q_offset=off, threads=1)
    for i in range(Tq):
        p = off + i
        keys = list(range(max(0, p - w + 1), min(Tk, p + 1)))
        assert np.allclose(o[0, 0, i], v[0, 0, keys].mean(axis=0), rtol=0, atol=1e-14)
        assert abs(lse[0, 0, i] - math.log(len(keys))) <= 1e-14


def pin_constant_shift(orc):
    # Adding c to every logit of a row leaves o unchanged and moves lse by c;
    # with c = 800 an oracle that does not subtract the maximum overflows.
    r = _rng(8)
    q = r.standard_normal((1, 2, 5, 4))
    k = r.standard_normal((1, 1, 7, 4))
    v = r.standard_normal((1, 1, 7, 4))
    base = r.standard_normal((5, 7))
    o1, l1 = orc.attention(q, k, v, 0.6, causal=False, mask=base, mask_strides=(0, 0, 7, 1), threads=1)
    o2, l2 = orc.attention(q, k, v, 0.6, causal=False, mask=base + 800.0, mask_strides=(0, 0, 7, 1),
                           threads=1)
    assert np.all(np.isfinite(o2)), o2
    assert np.allclose(o1, o2, rtol=0, atol=1e-12)
    assert np.allclose(l2 - l1, 800.0, rtol=0, atol=1e-10)


def pin_shape_errors(orc):
    # section 4, shape_and_argument_errors: 6 heads on 4 KV heads and Hkv > H
    # are rejected, negative sizes too, and o is left alone.
    q = np.zeros((1, 6, 2, 4))
    kv = np.zeros((1, 6, 3, 4))  # sized for 6 heads so no read can leave it
    o = np.full((1 * 6 * 2 * 4,), 7.0)
    lse = np.full((12,), 7.0)
    st = orc.raw(q, kv, kv, o, lse, 1, 6, 4, 2, 3, 4, 1.0, 0, 0, 0, None, None, (0, 0, 0, 0), None, 1)
    assert st == 2 and np.all(o == 7.0) and np.all(lse == 7.0), st
    st = orc.raw(q, kv, kv, o, lse, 1, 2, 4, 2, 3, 4, 1.0, 0, 0, 0, None, None, (0, 0, 0, 0), None, 1)
    assert st == 2 and np.all(o == 7.0), st
    st = orc.raw(q, kv, kv, o, lse, 1, 2, 2, -1, 3, 4, 1.0, 0, 0, 0, None, None, (0, 0, 0, 0), None, 1)
    assert st == 1 and np.all(o == 7.0), st
    st = orc.raw(q, kv, kv, o, lse, 1, 2, 2, 2, 3, 4, 1.0, -1, 0, 0, None, None, (0, 0, 0, 0), None, 1)
    assert st == 1 and np.all(o == 7.0), st


# ----------------------------------------------------------------------------
# Library cross-check, brute force over the flag space on tiny shapes
# ----------------------------------------------------------------------------

def _visible_ranges(Tq, Tk, causal, window, q_offset):
    """Visible keys of each row, enumerated as an index range."""
    out = []
    for i in range(Tq):
        p = q_offset + i
        hi = Tk if not causal else min(Tk, p + 1)
        lo = 0 if window <= 0 else max(0, p - window + 1)
        out.append(range(lo, max(lo, hi)))
    return out


def library_reference(q, k, v, scale, causal, window, q_offset, sinks, mask4):
    """float64 torch SDPA + logsumexp on a materialised additive mask; the sink
    is one extra key with a zero key vector, a zero value and mask z_h.
    ``mask4`` is the dense [B,Hq,Tq,Tk] additive mask or None."""
    B, Hq, Tq, D = q.shape
    Hkv, Tk = k.shape[1], k.shape[2]
    tq = torch.from_numpy(q)
    tk = torch.from_numpy(k).repeat_interleave(Hq // Hkv, dim=1)
    tv = torch.from_numpy(v).repeat_interleave(Hq // Hkv, dim=1)
    add = torch.full((B, Hq, Tq, Tk), -math.inf, dtype=torch.float64)
    for i, rng_ in enumerate(_visible_ranges(Tq, Tk, causal, window, q_offset)):
        for j in rng_:
            add[:, :, i, j] = 0.0
    if mask4 is not None:
        add = add + torch.from_numpy(mask4)
    if sinks is not None:
        tk = torch.cat([tk, torch.zeros(B, Hq, 1, D, dtype=torch.float64)], dim=2)
        tv = torch.cat([tv, torch.zeros(B, Hq, 1, D, dtype=torch.float64)], dim=2)
        zcol = torch.from_numpy(np.asarray(sinks, dtype=np.float64)).view(1, Hq, 1, 1).expand(B, Hq, Tq, 1)
        add = torch.cat([add, zcol], dim=3)
    if add.shape[-1] == 0:
        return np.zeros((B, Hq, Tq, D)), np.full((B, Hq, Tq), -np.inf)
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=add, scale=scale)
    lse = torch.logsumexp(scale * (tq @ tk.transpose(-1, -2)) + add, dim=-1)
    empty = torch.isneginf(add).all(dim=-1)
    o = torch.where(empty[..., None], torch.zeros_like(o), o)
    return o.numpy(), lse.numpy()


def pin_library_crosscheck(orc):
    r = _rng(9)
    heads = [(6, 2), (3, 1), (2, 2)]
    lens = [(0, 0), (1, 1), (2, 3), (3, 3), (5, 5), (17, 17), (4, 37), (37, 37)]
    n = 0
    for (Hq, Hkv), (Tq, Tk), causal, window, q_offset, use_sink, use_mask in itertools.product(
            heads, lens, (False, True), (0, 1, 3, 6), (0, 1, 24), (False, True), (False, True)):
        if causal and q_offset + Tq > Tk + 24:
            continue
        n += 1
        if n % 3:  # a third of the product keeps the run short but covers every factor
            continue
        B, D = 2, 4
        scale = 0.37
        q = r.standard_normal((B, Hq, Tq, D))
        k = r.standard_normal((B, Hkv, Tk, D))
        v = r.standard_normal((B, Hkv, Tk, D))
        sinks = r.standard_normal(Hq) if use_sink else None
        mask4 = None
        mask_flat, strides = None, (0, 0, 0, 0)
        if use_mask:
            # full [B,Hq,Tq,Tk] mask with some -inf entries
            m = r.standard_normal((B, Hq, Tq, Tk))
            m[r.random((B, Hq, Tq, Tk)) < 0.2] = -np.inf
            mask4 = m
            mask_flat = m.reshape(-1)
            strides = (Hq * Tq * Tk, Tq * Tk, Tk, 1)
        o, lse = orc.attention(q, k, v, scale, causal=causal, window=window, q_offset=q_offset,
                               sinks=sinks, mask=mask_flat, mask_strides=strides, threads=2)
        eo, else_ = library_reference(q, k, v, scale, causal, window, q_offset, sinks, mask4)
        ctx = (Hq, Hkv, Tq, Tk, causal, window, q_offset, use_sink, use_mask)
        assert np.allclose(o, eo, rtol=0, atol=1e-12), ctx
        same_inf = np.isneginf(lse) == np.isneginf(else_)
        assert np.all(same_inf), ctx
        fin = ~np.isneginf(else_)
        assert np.allclose(lse[fin], else_[fin], rtol=0, atol=1e-12), ctx


def pin_mask_strides(orc):
    # A square, non-symmetric mask stored three ways: dense [B,H,T,T],
    # broadcast [T,T] with strides (0,0,T,1), and transposed storage [T,T]
    # with strides (0,0,1,T).  All must agree with the library reference.
    r = _rng(10)
    B, Hq, Hkv, T, D = 2, 4, 2, 9, 5
    q = r.standard_normal((B, Hq, T, D))
    k = r.standard_normal((B, Hkv, T, D))
    v = r.standard_normal((B, Hkv, T, D))
    m = r.standard_normal((T, T)) * 2.0
    m[r.random((T, T)) < 0.3] = -np.inf
    m4 = np.broadcast_to(m, (B, Hq, T, T)).copy()
    eo, el = library_reference(q, k, v, 0.8, False, 0, 0, None, m4)
    for flat, strides in [(m4.reshape(-1), (Hq * T * T, T * T, T, 1)),
                          (m.reshape(-1), (0, 0, T, 1)),
                          (m.T.copy().reshape(-1), (0, 0, 1, T))]:
        o, lse = orc.attention(q, k, v, 0.8, causal=False, mask=flat, mask_strides=strides, threads=1)
        assert np.allclose(o, eo, rtol=0, atol=1e-12), strides
        fin = ~np.isneginf(el)
        assert np.array_equal(np.isneginf(lse), ~fin)
        assert np.allclose(lse[fin], el[fin], rtol=0, atol=1e-12), strides


def pin_row_subset_and_threads(orc):
    # The row-sampled entry and any thread count give the full run's bits.
    r = _rng(11)
    q = r.standard_normal((2, 4, 23, 8))
    k = r.standard_normal((2, 2, 30, 8))
    v = r.standard_normal((2, 2, 30, 8))
    o1, l1 = orc.attention(q, k, v, 0.5, causal=True, q_offset=7, threads=1)
    o8, l8 = orc.attention(q, k, v, 0.5, causal=True, q_offset=7, threads=8)
    assert np.array_equal(o1, o8) and np.array_equal(l1, l8)
    rows = np.array([0, 5, 22, 11])
    orr, lr = orc.attention(q, k, v, 0.5, causal=True, q_offset=7, rows=rows, threads=3)
    assert np.array_equal(orr, o1[:, :, rows]) and np.array_equal(lr, l1[:, :, rows])


ALL_PINS = [
    pin_worked_example,
    pin_sink_identity,
    pin_sink_weights_sum,
    pin_weights_sum_to_one,
    pin_empty_rows,
    pin_single_key,
    pin_window_one,
    pin_zero_query_uniform,
    pin_constant_shift,
    pin_shape_errors,
    pin_library_crosscheck,
    pin_mask_strides,
    pin_row_subset_and_threads,
]
