"""Host-side checks of the C ABI: the library loads, exports what
include/fa.h declares, and rejects bad arguments before touching anything.

No GPU is needed: every call below fails validation (or is a no-op) before
any CUDA call, and ``o``/``lse`` are host canary buffers that must stay
untouched ("FlashAttention forward in C", section 4: errors before any write).
"""
import ctypes
import re
import subprocess
from pathlib import Path

import numpy as np
import pytest

import exact_tiled_attention_flashattention_gb300 as fa

ROOT = Path(__file__).resolve().parent.parent


def _declared_functions():
    text = (ROOT / "include" / "fa.h").read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    return fa.load()


def test_library_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert "fa_fwd" in names and "fa_last_error" in names
    out = subprocess.run(["nm", "-D", "--defined-only", str(fa.library_path())], capture_output=True, text=True,
                         check=True).stdout
    exported = set(line.split()[-1] for line in out.splitlines() if line.strip())
    for n in names:
        assert n in exported, n
        assert hasattr(lib, n), n


def test_version(lib):
    assert fa.fa_version() >= 100


class Canary:
    """Host buffers standing in for o and lse; any write would show."""

    def __init__(self, n=4096):
        self.o = np.full(n, 12345.0, dtype=np.float32)
        self.lse = np.full(n, 6789.0, dtype=np.float32)
        self.q = np.zeros(n, dtype=np.float32)

    def ptrs(self):
        return self.q.ctypes.data, self.o.ctypes.data, self.lse.ctypes.data

    def untouched(self):
        return bool(np.all(self.o == 12345.0) and np.all(self.lse == 6789.0))


def _call(c, **kw):
    q, o, lse = c.ptrs()
    args = dict(q=q, k=q, v=q, o=o, lse=lse, B=1, Hq=2, Hkv=1, Tq=4, Tk=4, d=8, scale=0.5, q_offset=0, causal=1,
                window=0, sinks=None, mask=None, mask_sb=0, mask_sh=0, mask_sq=0, mask_sk=0, dtype=fa.FA_DTYPE_F32)
    args.update(kw)
    return fa.fa_fwd(args["q"], args["k"], args["v"], args["o"], args["lse"], args["B"], args["Hq"], args["Hkv"],
                     args["Tq"], args["Tk"], args["d"], args["scale"], args["q_offset"], args["causal"],
                     args["window"], args["sinks"], args["mask"], args["mask_sb"], args["mask_sh"], args["mask_sq"],
                     args["mask_sk"], args["dtype"], 0, check=False)


CASES = [
    ("unknown dtype", dict(dtype=7), fa.FA_EINVAL),
    ("negative B", dict(B=-1), fa.FA_EINVAL),
    ("negative Tq", dict(Tq=-3), fa.FA_EINVAL),
    ("negative Tk", dict(Tk=-1), fa.FA_EINVAL),
    ("negative d", dict(d=-8), fa.FA_EINVAL),
    ("negative q_offset", dict(q_offset=-1), fa.FA_EINVAL),
    ("nan scale", dict(scale=float("nan")), fa.FA_EINVAL),
    ("inf scale", dict(scale=float("inf")), fa.FA_EINVAL),
    ("null q", dict(q=None), fa.FA_EINVAL),
    ("null o", dict(o=None), fa.FA_EINVAL),
    ("null k with Tk > 0", dict(k=None), fa.FA_EINVAL),
    ("null v with Tk > 0", dict(v=None), fa.FA_EINVAL),
    ("negative mask stride", dict(mask=1 << 20, mask_sq=-4), fa.FA_EINVAL),
    ("overflowing sizes", dict(B=1 << 40, Hq=1 << 20, Hkv=1 << 20, Tq=1 << 20), fa.FA_EINVAL),
    ("6 heads on 4 KV heads", dict(Hq=6, Hkv=4), fa.FA_ESHAPE),
    ("Hkv > Hq", dict(Hq=2, Hkv=4), fa.FA_ESHAPE),
    ("Hkv = 0", dict(Hkv=0), fa.FA_ESHAPE),
    ("odd d", dict(d=7), fa.FA_EUNSUPPORTED),
    ("zero d", dict(d=0), fa.FA_EUNSUPPORTED),
    ("fp32 d > 256", dict(d=258), fa.FA_EUNSUPPORTED),
    ("bf16 d = 100 (not a multiple of 8)", dict(d=100, dtype=fa.FA_DTYPE_BF16), fa.FA_EUNSUPPORTED),
    ("bf16 d = 136 (> 128)", dict(d=136, dtype=fa.FA_DTYPE_BF16), fa.FA_EUNSUPPORTED),
    ("fp32 tc d = 30 (not a multiple of 4)", dict(d=30, dtype=fa.FA_DTYPE_F32_TC), fa.FA_EUNSUPPORTED),
    ("fp32 tc d = 132 (> 128)", dict(d=132, dtype=fa.FA_DTYPE_F32_TC), fa.FA_EUNSUPPORTED),
    ("unknown dtype 4", dict(dtype=4), fa.FA_EINVAL),
    ("e4m3 d = 24 (not a multiple of 16)", dict(d=24, dtype=fa.FA_DTYPE_FP8_E4M3), fa.FA_EUNSUPPORTED),
    ("e4m3 d = 144 (> 128)", dict(d=144, dtype=fa.FA_DTYPE_FP8_E4M3), fa.FA_EUNSUPPORTED),
    ("Tk >= 2^30", dict(Tk=1 << 30), fa.FA_EUNSUPPORTED),
    ("Tq >= 2^30", dict(Tq=1 << 30, B=1, Hq=1, Hkv=1, d=2), fa.FA_EUNSUPPORTED),
]


@pytest.mark.parametrize("name,kw,expected", CASES, ids=[c[0] for c in CASES])
def test_rejected_before_any_write(lib, name, kw, expected):
    c = Canary()
    st = _call(c, **kw)
    assert st == expected, (name, st, fa.fa_last_error())
    assert fa.fa_last_error(), "a non-OK status must leave a message"
    assert c.untouched()


def test_unaligned_pointer_rejected(lib):
    c = Canary()
    q, o, lse = c.ptrs()
    st = _call(c, q=q + 4)
    assert st == fa.FA_EUNSUPPORTED and c.untouched()
    st = _call(c, o=o + 8)
    assert st == fa.FA_EUNSUPPORTED and c.untouched()


@pytest.mark.parametrize("kw", [dict(Tq=0), dict(B=0), dict(Hq=0, Hkv=0)])
def test_empty_problem_is_a_no_op(lib, kw):
    c = Canary()
    st = _call(c, **kw)
    assert st == fa.FA_OK and c.untouched()


def test_binding_raises_on_error(lib):
    c = Canary()
    q, o, lse = c.ptrs()
    with pytest.raises(fa.FaError) as ei:
        fa.fa_fwd(q, q, q, o, lse, 1, 6, 4, 4, 4, 8, 0.5, 0, 1, 0, None, None, 0, 0, 0, 0, fa.FA_DTYPE_F32, 0)
    assert ei.value.status == fa.FA_ESHAPE
    assert c.untouched()


# ---------------------------------------------------------------- strided

def _strided(fa_mod, **kw):
    """fa_fwd_strided on fake (aligned, never dereferenced) pointers: every
    case below is rejected before any launch."""
    a = dict(B=2, Hq=4, Hkv=2, Tq=8, Tk=8, d=64, dtype=fa_mod.FA_DTYPE_BF16)
    a.update(kw)
    B, Hq, Hkv, Tq, Tk, d = a["B"], a["Hq"], a["Hkv"], a["Tq"], a["Tk"], a["d"]
    qs = a.get("qs", (Hq * Tq * d, Tq * d, d))
    ks = a.get("ks", (Hkv * Tk * d, Tk * d, d))
    os_ = a.get("os", qs)
    p = 1 << 20  # 16-byte aligned fake address
    return fa_mod.fa_fwd_strided(p, p, p, p, None, B, Hq, Hkv, Tq, Tk, d, qs, ks, ks, os_, 0.125, 0, 1, 0, None,
                                 None, 0, 0, 0, 0, a["dtype"], 0, check=False)


@pytest.mark.parametrize("case,kw,want", [
    ("negative row stride", dict(qs=(2048, 512, -64)), "FA_EINVAL"),
    ("output rows overlap", dict(os=(2048, 512, 32)), "FA_EINVAL"),
    ("output heads overlap", dict(os=(2048, 64, 64)), "FA_EINVAL"),
    ("bf16 stride not a multiple of 8", dict(qs=(2048, 516, 64), os=(4096, 1024, 128)), "FA_EUNSUPPORTED"),
    ("bf16 zero batch stride on k", dict(ks=(0, 512, 64)), "FA_EUNSUPPORTED"),
    ("fp32 odd stride", dict(dtype=1 - 1, qs=(2048, 513, 64), os=(4096, 1024, 128)), "FA_EUNSUPPORTED"),
    ("fp32 tc stride not a multiple of 4", dict(dtype=2, qs=(2048, 514, 64), os=(4096, 1024, 128)),
     "FA_EUNSUPPORTED"),
    ("fp32 tc zero batch stride on k", dict(dtype=2, ks=(0, 512, 64)), "FA_EUNSUPPORTED"),
    ("e4m3 stride not a multiple of 16", dict(dtype=3, qs=(2048, 520, 64), os=(4096, 1024, 128)),
     "FA_EUNSUPPORTED"),
])
def test_strided_rejections(lib, case, kw, want):
    import exact_tiled_attention_flashattention_gb300 as fa_mod
    assert _strided(fa_mod, **kw) == getattr(fa_mod, want), case
    assert fa_mod.fa_last_error() != ""


def test_strided_bshd_layout_is_valid_up_to_launch(lib):
    # A [B, T, H, d] layout passes validation; with B*Hq*Tq == 0 the call is
    # a no-op (nothing is launched on this GPU-less host).
    import exact_tiled_attention_flashattention_gb300 as fa_mod
    B, T, H, d = 2, 8, 4, 64
    st = _strided(fa_mod, Tq=0, qs=(T * H * d, d, H * d), ks=(T * 2 * d, d, 2 * d))
    assert st == fa_mod.FA_OK


# ---------------------------------------------------------------- paged

@pytest.mark.parametrize("case,kw,want", [
    ("fp32 is not paged", dict(dtype=0), "FA_EUNSUPPORTED"),
    ("fp32 tc is not paged", dict(dtype=2), "FA_EUNSUPPORTED"),
    ("e4m3 is not paged", dict(dtype=3), "FA_EUNSUPPORTED"),
    ("group * Tq > 128", dict(Tq=65), "FA_EUNSUPPORTED"),
    ("page size 48", dict(page_size=48), "FA_EUNSUPPORTED"),
    ("page size 4", dict(page_size=4), "FA_EUNSUPPORTED"),
    ("table too short", dict(max_blocks=2), "FA_EINVAL"),
    ("null seq_lens", dict(seq_lens=None), "FA_EINVAL"),
    ("negative pages", dict(num_pages=-1), "FA_EINVAL"),
    ("Hq % Hkv", dict(Hq=6, Hkv=4), "FA_ESHAPE"),
])
def test_paged_rejections(lib, case, kw, want):
    import exact_tiled_attention_flashattention_gb300 as fa_mod
    a = dict(B=2, Hq=4, Hkv=2, Tq=1, d=64, seq_lens=1 << 20, max_seq_len=1000, max_blocks=16, page_size=64,
             num_pages=40, dtype=fa_mod.FA_DTYPE_BF16)
    a.update(kw)
    p = 1 << 20
    st = fa_mod.fa_fwd_paged(p, p, p, p, None, a["B"], a["Hq"], a["Hkv"], a["Tq"], a["d"], a["seq_lens"],
                             a["max_seq_len"], p, a["max_blocks"], a["page_size"], a["num_pages"], 0.125, 1, 0, None,
                             a["dtype"], 0, check=False)
    assert st == getattr(fa_mod, want), case


# ---------------------------------------------------------------- varlen

@pytest.mark.parametrize("case,kw,want", [
    ("null cu_seqlens_q", dict(cuq=None), "FA_EINVAL"),
    ("max_seqlen_q > total_q", dict(max_q=300), "FA_EUNSUPPORTED"),
    ("overlapping output rows", dict(o_st=32), "FA_EINVAL"),
    ("Hq % Hkv", dict(Hq=6, Hkv=4), "FA_ESHAPE"),
    ("bf16 d = 100", dict(d=100), "FA_EUNSUPPORTED"),
    ("fp32 tc is not varlen", dict(dtype=2), "FA_EUNSUPPORTED"),
    ("e4m3 varlen d = 24", dict(dtype=3, d=24), "FA_EUNSUPPORTED"),
])
def test_varlen_rejections(lib, case, kw, want):
    import exact_tiled_attention_flashattention_gb300 as fa_mod
    a = dict(B=3, Hq=4, Hkv=2, d=64, cuq=1 << 20, total_q=200, total_k=200, max_q=100, max_k=100, o_st=None,
             dtype=fa_mod.FA_DTYPE_BF16)
    a.update(kw)
    p = 1 << 20
    H, d = a["Hq"], a["d"]
    qs, ks = (d, H * d), (d, a["Hkv"] * d)
    os_ = (d, a["o_st"]) if a["o_st"] is not None else qs
    st = fa_mod.fa_fwd_varlen(p, p, p, p, None, a["B"], a["Hq"], a["Hkv"], d, a["cuq"], p, a["total_q"],
                              a["total_k"], a["max_q"], a["max_k"], qs, ks, ks, os_, 0.125, 1, 0, None, a["dtype"], 0,
                              check=False)
    assert st == getattr(fa_mod, want), case


def test_grid_cap_hook_checks_its_argument(lib):
    """fa_test_max_ctas rejects a negative cap before changing anything and
    accepts 0 (off) and positive caps; no GPU is touched."""
    assert lib.fa_test_max_ctas(-1) == fa.FA_EINVAL
    assert b"negative" in lib.fa_last_error()
    assert lib.fa_test_max_ctas(7) == fa.FA_OK
    assert lib.fa_test_max_ctas(0) == fa.FA_OK
