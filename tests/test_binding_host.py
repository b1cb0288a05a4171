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
