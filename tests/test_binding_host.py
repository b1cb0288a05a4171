"""Host checks of the Python binding: it fails loudly instead of falling back.

No GPU is needed: the checks run before any call reaches the library.  A
missing libfa.so raises ImportError (there is no CPU path to fall back to);
host tensors are refused before their addresses could reach the kernels; the
float32 side inputs (sinks, mask, lse) are checked for dtype and size.
"""
from __future__ import annotations

import pytest
import torch

import exact_tiled_attention_flashattention_gb300 as fa


def test_missing_library_raises(monkeypatch, tmp_path):
    monkeypatch.setattr(fa, "_LIB_PATH", tmp_path / "libfa.so")
    monkeypatch.setattr(fa, "_lib", None)
    with pytest.raises(ImportError, match="build the CUDA library"):
        fa.fa_version()
    with pytest.raises(ImportError):
        fa.fa_fwd(None, None, None, None, None, 0, 0, 0, 0, 0, 0, 1.0, 0, 0, 0, None, None, 0, 0, 0, 0,
                  fa.FA_DTYPE_BF16, 0)


def _qkv(dtype=torch.bfloat16):
    q = torch.zeros((1, 2, 8, 64), dtype=dtype)
    k = torch.zeros((1, 1, 8, 64), dtype=dtype)
    return q, k, k.clone()


def test_host_tensors_are_refused(monkeypatch):
    called = []
    monkeypatch.setattr(fa, "load", lambda: called.append(1))
    q, k, v = _qkv()
    with pytest.raises(ValueError, match="CUDA tensor"):
        fa.attention(q, k, v)
    with pytest.raises(ValueError, match="CUDA tensor"):
        fa.varlen_attention(q[0].transpose(0, 1), k[0].transpose(0, 1), v[0].transpose(0, 1),
                            torch.tensor([0, 8], dtype=torch.int32), torch.tensor([0, 8], dtype=torch.int32), 8, 8)
    kc = torch.zeros((4, 16, 1, 64), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        fa.paged_attention(q, kc, kc, torch.zeros((1, 4), dtype=torch.int32), torch.tensor([8], dtype=torch.int32),
                           8)
    assert called == []  # nothing reached the library


def test_tensor_device_check():
    dev = torch.device("cuda", 0)  # a device object needs no GPU
    with pytest.raises(ValueError, match="k must be a CUDA tensor on cuda:0"):
        fa._check_tensors(dev, k=torch.zeros(1))
    fa._check_tensors(dev, k=None, mask=1 << 20)  # absent arguments and raw device addresses pass
    with pytest.raises(ValueError, match="q must be a CUDA tensor"):
        fa._check_tensors(torch.device("cpu"))


def test_float32_side_inputs():
    with pytest.raises(TypeError, match="sinks must be float32"):
        fa._check_f32("sinks", torch.zeros(4, dtype=torch.bfloat16), 4)
    with pytest.raises(ValueError, match="at least 4 elements"):
        fa._check_f32("sinks", torch.zeros(3), 4)
    fa._check_f32("sinks", torch.zeros(4), 4)
    fa._check_f32("mask", None)
    fa._check_f32("mask", 1 << 20)


# --- the binding's argument lists against include/fa.h -------------------------

def _header_signatures():
    """{name: [C parameter types]} of every function include/fa.h declares."""
    import re
    from pathlib import Path
    src = (Path(__file__).resolve().parents[1] / "include" / "fa.h").read_text()
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    sigs = {}
    for name, params in re.findall(r"\b(fa_\w+)\s*\(([^()]*)\)\s*;", src):
        params = " ".join(params.split())
        if params in ("", "void"):
            sigs[name] = []
            continue
        types = []
        for p in params.split(","):
            p = p.strip()
            if "*" in p:
                types.append("ptr")
            else:
                types.append(p.rsplit(" ", 1)[0].replace("const ", "").strip())
        sigs[name] = types
    return sigs


def test_ctypes_argument_lists_match_the_header():
    import ctypes
    lib = fa.load()
    want = {"ptr": ctypes.c_void_p, "int64_t": ctypes.c_int64, "int": ctypes.c_int, "float": ctypes.c_float,
            "size_t": ctypes.c_size_t}
    sigs = _header_signatures()
    assert {"fa_fwd", "fa_fwd_strided", "fa_fwd_paged", "fa_fwd_varlen", "fa_last_error", "fa_version",
            "fa_device_status", "fa_test_drop_arrive", "fa_fwd_splitkv", "fa_splitkv_workspace_bytes"} <= set(sigs)
    for name, types in sigs.items():
        got = getattr(lib, name).argtypes
        assert got is not None, name
        assert [want[t] for t in types] == list(got), name


# --- what the tensor wrappers pass on ------------------------------------------

def _recording(monkeypatch, entry):
    """Let host tensors through the device check and record the raw call."""
    import contextlib
    calls = []
    monkeypatch.setattr(fa, "_check_tensors", lambda dev, **kw: None)
    monkeypatch.setattr(torch.cuda, "device", lambda dev: contextlib.nullcontext())
    monkeypatch.setattr(fa, entry, lambda *a, **kw: calls.append(a))
    return calls


def test_attention_marshals_a_strided_view(monkeypatch):
    calls = _recording(monkeypatch, "fa_fwd_strided")
    B, Hq, Hkv, T, d = 2, 4, 2, 8, 64
    q = torch.zeros((B, T, Hq, d), dtype=torch.bfloat16).transpose(1, 2)  # [B, H, T, d] view of BSHD storage
    k = torch.zeros((B, Hkv, T, d), dtype=torch.bfloat16)
    z = torch.zeros(Hq)
    o, lse = fa.attention(q, k, k, q_offset=3, window=5, sinks=z)
    (a,) = calls
    assert a[5:11] == (B, Hq, Hkv, T, T, d)
    assert a[11] == (T * Hq * d, d, Hq * d)  # q: batch, head, row strides of the view
    assert a[12] == (Hkv * T * d, T * d, d)
    assert a[14] == tuple(o.stride()[:3]) and o.dtype == torch.bfloat16 and lse.dtype == torch.float32
    assert a[15] == pytest.approx(d ** -0.5)
    assert a[16:21] == (3, True, 5, z, None)
    assert a[25] == fa.FA_DTYPE_BF16
    fa.attention(q.float(), k.float(), k.float(), fp32_tc=True)
    assert calls[1][25] == fa.FA_DTYPE_F32_TC
    fa.attention(q.float(), k.float(), k.float())
    assert calls[2][25] == fa.FA_DTYPE_F32


def test_attention_rejects_bad_arguments(monkeypatch):
    _recording(monkeypatch, "fa_fwd_strided")
    q = torch.zeros((1, 2, 8, 64), dtype=torch.bfloat16)
    k = torch.zeros((1, 1, 8, 64), dtype=torch.bfloat16)
    with pytest.raises(TypeError, match="share a dtype"):
        fa.attention(q, k.float(), k.float())
    with pytest.raises(TypeError, match="sinks must be float32"):
        fa.attention(q, k, k, sinks=torch.zeros(2, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="at least 2 elements"):
        fa.attention(q, k, k, sinks=torch.zeros(1))
    with pytest.raises(ValueError, match="lse_out"):
        fa.attention(q, k, k, lse_out=torch.zeros((1, 2, 8), dtype=torch.float64))
    with pytest.raises(ValueError, match="last dimension contiguous"):
        fa.attention(q.transpose(2, 3), k, k)


def test_varlen_and_paged_marshal(monkeypatch):
    calls = _recording(monkeypatch, "fa_fwd_varlen")
    q = torch.zeros((30, 4, 64), dtype=torch.bfloat16)
    k = torch.zeros((40, 2, 64), dtype=torch.bfloat16)
    cq = torch.tensor([0, 10, 30], dtype=torch.int32)
    ck = torch.tensor([0, 15, 40], dtype=torch.int32)
    o, lse = fa.varlen_attention(q, k, k, cq, ck, 20, 25, causal=True)
    (a,) = calls
    assert a[5:9] == (2, 4, 2, 64) and a[11:15] == (30, 40, 20, 25)
    assert a[15] == (64, 4 * 64) and a[16] == (64, 2 * 64)  # (head, row) strides
    assert o.shape == (30, 4, 64) and lse.shape == (4, 30)
    with pytest.raises(ValueError, match="B \\+ 1"):
        fa.varlen_attention(q, k, k, cq, ck[:2], 20, 25)

    calls = _recording(monkeypatch, "fa_fwd_paged")
    qd = torch.zeros((3, 4, 1, 64), dtype=torch.bfloat16)
    kc = torch.zeros((10, 16, 2, 64), dtype=torch.bfloat16)
    table = torch.zeros((3, 5), dtype=torch.int32)
    sl = torch.tensor([20, 33, 80], dtype=torch.int32)
    fa.paged_attention(qd, kc, kc, table, sl, 80)
    (a,) = calls
    assert a[5:10] == (3, 4, 2, 1, 64)
    assert a[11] == 80 and a[13:16] == (5, 16, 10)
    assert a[20] == fa.FA_DTYPE_BF16
