"""Python binding of libfa (the C ABI declared in include/fa.h).

Argument marshalling only: every step of the attention forward runs in the
CUDA kernels of ``libfa.so``.  There is no CPU fallback; importing the binding
without the built library raises.

``fa_fwd`` mirrors the C entry point name for name.  Tensor arguments may be
torch tensors (their ``data_ptr()`` is passed) or integer device addresses;
``stream`` may be a ``torch.cuda.Stream``, an integer handle or None (the
current torch stream).  ``attention`` is a convenience wrapper that allocates
``o`` and ``lse`` with torch and calls ``fa_fwd``.
"""
from __future__ import annotations

import ctypes
from pathlib import Path

__all__ = ["FA_OK", "FA_EINVAL", "FA_ESHAPE", "FA_EUNSUPPORTED", "FA_ECUDA", "FA_ETIMEOUT", "FA_DTYPE_F32",
           "FA_DTYPE_BF16", "FA_DTYPE_F32_TC", "FA_DTYPE_FP8_E4M3", "FaError", "fa_fwd", "fa_last_error",
           "fa_version", "fa_device_status", "fa_test_drop_arrive", "fa_test_max_ctas", "attention", "fa_fwd_splitkv", "fa_splitkv_workspace_bytes", "fa_fwd_splitkv_noalloc",
           "splitkv_attention", "library_path", "load"]

FA_OK, FA_EINVAL, FA_ESHAPE, FA_EUNSUPPORTED, FA_ECUDA, FA_ETIMEOUT = 0, 1, 2, 3, 4, 5
FA_DTYPE_F32, FA_DTYPE_BF16, FA_DTYPE_F32_TC, FA_DTYPE_FP8_E4M3 = 0, 1, 2, 3
_STATUS = {0: "FA_OK", 1: "FA_EINVAL", 2: "FA_ESHAPE", 3: "FA_EUNSUPPORTED", 4: "FA_ECUDA", 5: "FA_ETIMEOUT"}

_LIB_PATH = Path(__file__).resolve().parent / "libfa.so"
_lib = None


class FaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_STATUS.get(status, status)}: {message}")
        self.status = status


def library_path() -> Path:
    return _LIB_PATH


def load():
    """Load libfa.so (built by the repository's build step) and declare its
    signatures.  Raises if the library has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not _LIB_PATH.exists():
        raise ImportError(f"{_LIB_PATH} is missing: build the CUDA library first "
                          "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(str(_LIB_PATH))
    i64, vp = ctypes.c_int64, ctypes.c_void_p
    lib.fa_fwd.restype = ctypes.c_int
    lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, ctypes.c_float, i64, ctypes.c_int,
                           i64, vp, vp, i64, i64, i64, i64, ctypes.c_int, vp]
    lib.fa_fwd_strided.restype = ctypes.c_int
    lib.fa_fwd_strided.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64] + [i64] * 12 + [
        ctypes.c_float, i64, ctypes.c_int, i64, vp, vp, i64, i64, i64, i64, ctypes.c_int, vp]
    lib.fa_fwd_paged.restype = ctypes.c_int
    lib.fa_fwd_paged.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, vp, i64, vp, i64, i64, i64,
                                 ctypes.c_float, ctypes.c_int, i64, vp, ctypes.c_int, vp]
    lib.fa_fwd_varlen.restype = ctypes.c_int
    lib.fa_fwd_varlen.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, vp, vp, i64, i64, i64, i64] + [i64] * 8 + [
        ctypes.c_float, ctypes.c_int, i64, vp, ctypes.c_int, vp]
    lib.fa_fwd_splitkv.restype = ctypes.c_int
    lib.fa_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, ctypes.c_float, i64,
                                   ctypes.c_int, i64, vp, vp, i64, i64, i64, i64, vp, ctypes.c_size_t, ctypes.c_int,
                                   vp]
    lib.fa_fwd_splitkv_noalloc.restype = ctypes.c_int
    lib.fa_fwd_splitkv_noalloc.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, ctypes.c_float, i64,
                                           ctypes.c_int, i64, vp, vp, i64, i64, i64, i64, ctypes.c_int, vp]
    lib.fa_splitkv_workspace_bytes.restype = ctypes.c_int
    lib.fa_splitkv_workspace_bytes.argtypes = [i64, i64, i64, i64, i64, ctypes.c_int, vp]
    lib.fa_last_error.restype = ctypes.c_char_p
    lib.fa_last_error.argtypes = []
    lib.fa_version.restype = ctypes.c_int
    lib.fa_version.argtypes = []
    lib.fa_device_status.restype = ctypes.c_int
    lib.fa_device_status.argtypes = [vp]
    lib.fa_test_drop_arrive.restype = ctypes.c_int
    lib.fa_test_drop_arrive.argtypes = [ctypes.c_int]
    lib.fa_test_max_ctas.restype = ctypes.c_int
    lib.fa_test_max_ctas.argtypes = [ctypes.c_int64]
    _lib = lib
    return lib


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x or None
    return x.data_ptr() or None


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream or None
    if isinstance(s, int):
        return s or None
    return s.cuda_stream or None


def _check_tensors(dev, **tensors):
    """The tensor wrappers pass raw addresses to the kernels, so every tensor
    argument must live on the CUDA device ``dev`` (a host tensor's address
    would reach the kernels as if it were device memory).  Integers (device
    addresses) and None pass through."""
    if dev.type != "cuda":
        raise ValueError(f"q must be a CUDA tensor (got one on {dev})")
    for name, t in tensors.items():
        if t is None or isinstance(t, int):
            continue
        if t.device != dev:
            raise ValueError(f"{name} must be a CUDA tensor on {dev} (got one on {t.device})")


def _check_f32(name, t, min_numel=0):
    """sinks and mask are read as float32 by the kernels."""
    import torch
    if t is None or isinstance(t, int):
        return
    if t.dtype != torch.float32:
        raise TypeError(f"{name} must be float32 (got {t.dtype})")
    if t.numel() < min_numel:
        raise ValueError(f"{name} must hold at least {min_numel} elements (got {t.numel()})")


def fa_last_error() -> str:
    return load().fa_last_error().decode()


def fa_version() -> int:
    return load().fa_version()


def fa_device_status(stream=None, *, check=True) -> int:
    """fa_device_status: FA_ETIMEOUT if a bounded wait in a tensor-core kernel
    ran out since the previous check (raised as FaError when ``check``)."""
    lib = load()
    st = lib.fa_device_status(_stream(stream))
    if check and st != FA_OK:
        raise FaError(st, lib.fa_last_error().decode())
    return st


def fa_test_drop_arrive(enable: bool) -> int:
    """Test hook: while enabled, CTA 0 of each tensor-core kernel skips one load."""
    lib = load()
    st = lib.fa_test_drop_arrive(1 if enable else 0)
    if st != FA_OK:
        raise FaError(st, lib.fa_last_error().decode())
    return st


def fa_test_max_ctas(n: int) -> int:
    """Test hook: cap the persistent tensor-core launches at ``n`` CTAs (0: off)."""
    lib = load()
    st = lib.fa_test_max_ctas(int(n))
    if st != FA_OK:
        raise FaError(st, lib.fa_last_error().decode())
    return st


def fa_fwd(q, k, v, o, lse, B, Hq, Hkv, Tq, Tk, d, scale, q_offset, causal, window, sinks, mask, mask_sb,
           mask_sh, mask_sq, mask_sk, dtype, stream=None, *, check=True) -> int:
    """Call the C entry point; raises FaError on a non-OK status when ``check``."""
    lib = load()
    st = lib.fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(Hq), int(Hkv), int(Tq), int(Tk),
                    int(d), float(scale), int(q_offset), int(bool(causal)), int(window), _ptr(sinks), _ptr(mask),
                    int(mask_sb), int(mask_sh), int(mask_sq), int(mask_sk), int(dtype), _stream(stream))
    if check and st != FA_OK:
        raise FaError(st, lib.fa_last_error().decode())
    return st


def fa_fwd_strided(q, k, v, o, lse, B, Hq, Hkv, Tq, Tk, d, q_strides, k_strides, v_strides, o_strides, scale,
                   q_offset, causal, window, sinks, mask, mask_sb, mask_sh, mask_sq, mask_sk, dtype, stream=None, *,
                   check=True) -> int:
    """Call the strided C entry point (each *_strides = (batch, head, row) in
    elements, d contiguous); raises FaError on a non-OK status when ``check``."""
    lib = load()
    st = lib.fa_fwd_strided(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(Hq), int(Hkv), int(Tq),
                            int(Tk), int(d), *[int(x) for x in (*q_strides, *k_strides, *v_strides, *o_strides)],
                            float(scale), int(q_offset), int(bool(causal)), int(window), _ptr(sinks), _ptr(mask),
                            int(mask_sb), int(mask_sh), int(mask_sq), int(mask_sk), int(dtype), _stream(stream))
    if check and st != FA_OK:
        raise FaError(st, lib.fa_last_error().decode())
    return st


def fa_splitkv_workspace_bytes(B, Hq, Hkv, Tq, d, dtype) -> int:
    """Bytes of device workspace that fa_fwd_splitkv needs for these sizes on
    the current device (0 when the call takes the plain fa_fwd path)."""
    lib = load()
    n = ctypes.c_size_t(0)
    st = lib.fa_splitkv_workspace_bytes(int(B), int(Hq), int(Hkv), int(Tq), int(d), int(dtype), ctypes.addressof(n))
    if st != FA_OK:
        raise FaError(st, lib.fa_last_error().decode())
    return int(n.value)


def fa_fwd_splitkv(q, k, v, o, lse, B, Hq, Hkv, Tq, Tk, d, scale, q_offset, causal, window, sinks, mask, mask_sb,
                   mask_sh, mask_sq, mask_sk, workspace, workspace_bytes, dtype, stream=None, *, check=True) -> int:
    """Call the split-KV C entry point (contiguous tensors, a caller-owned
    device workspace); raises FaError on a non-OK status when ``check``."""
    lib = load()
    st = lib.fa_fwd_splitkv(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(Hq), int(Hkv), int(Tq),
                            int(Tk), int(d), float(scale), int(q_offset), int(bool(causal)), int(window), _ptr(sinks),
                            _ptr(mask), int(mask_sb), int(mask_sh), int(mask_sq), int(mask_sk), _ptr(workspace),
                            int(workspace_bytes), int(dtype), _stream(stream))
    if check and st != FA_OK:
        raise FaError(st, lib.fa_last_error().decode())
    return st


FA_SPLITKV_NOALLOC_MAX_SCRATCH = 4 << 20  # bytes of the library's static split-KV scratch per GPU


def fa_fwd_splitkv_noalloc(q, k, v, o, lse, B, Hq, Hkv, Tq, Tk, d, scale, q_offset, causal, window, sinks, mask,
                           mask_sb, mask_sh, mask_sq, mask_sk, dtype, stream=None, *, check=True) -> int:
    """Call the C entry point that runs split-KV with the library's static
    scratch array instead of a workspace (for callers that cannot allocate
    device memory); raises FaError on a non-OK status when ``check``."""
    lib = load()
    st = lib.fa_fwd_splitkv_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(Hq), int(Hkv),
                                    int(Tq), int(Tk), int(d), float(scale), int(q_offset), int(bool(causal)),
                                    int(window), _ptr(sinks), _ptr(mask), int(mask_sb), int(mask_sh), int(mask_sq),
                                    int(mask_sk), int(dtype), _stream(stream))
    if check and st != FA_OK:
        raise FaError(st, lib.fa_last_error().decode())
    return st


def splitkv_attention(q, k, v, *, scale=None, q_offset=0, causal=True, window=0, sinks=None, mask=None,
                      mask_strides=(0, 0, 0, 0), workspace=None, out=None, lse_out=None, stream=None):
    """Decode attention through fa_fwd_splitkv for contiguous bf16 CUDA
    tensors q [B,Hq,Tq,d], k/v [B,Hkv,Tk,d]; returns (o, lse).  ``workspace``
    is a uint8 CUDA tensor of at least fa_splitkv_workspace_bytes bytes (one
    is allocated with torch when None)."""
    import torch
    B, Hq, Tq, d = q.shape
    Hkv, Tk = k.shape[1], k.shape[2]
    _check_tensors(q.device, k=k, v=v, out=out, lse_out=lse_out, sinks=sinks, mask=mask, workspace=workspace)
    _check_f32("sinks", sinks, Hq)
    _check_f32("mask", mask)
    if q.dtype != torch.bfloat16 or k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k and v must be bfloat16")
    for name, t in (("q", q), ("k", k), ("v", v)) + ((("out", out),) if out is not None else ()):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    with torch.cuda.device(q.device):
        need = fa_splitkv_workspace_bytes(B, Hq, Hkv, Tq, d, FA_DTYPE_BF16)
        if workspace is None:
            workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
        nbytes = workspace.numel() * workspace.element_size()
        o = out if out is not None else torch.empty((B, Hq, Tq, d), dtype=torch.bfloat16, device=q.device)
        lse = lse_out if lse_out is not None else torch.empty((B, Hq, Tq), dtype=torch.float32, device=q.device)
        sc = (1.0 / d ** 0.5) if scale is None else scale
        fa_fwd_splitkv(q, k, v, o, lse, B, Hq, Hkv, Tq, Tk, d, sc, q_offset, causal, window, sinks, mask,
                       *mask_strides, workspace, nbytes, FA_DTYPE_BF16, stream)
    return o, lse


def attention(q, k, v, *, scale=None, q_offset=0, causal=True, window=0, sinks=None, mask=None,
              mask_strides=(0, 0, 0, 0), with_lse=True, out=None, lse_out=None, stream=None, fp32_tc=False):
    """o [B,Hq,Tq,d] (q's dtype; bf16 for e4m3 inputs) and lse [B,Hq,Tq] (fp32)
    for CUDA tensors q [B,Hq,Tq,d], k/v [B,Hkv,Tk,d] (fp32, bf16 or
    float8_e4m3fn).  The tensors may be
    strided views (a [B,T,H,d] buffer seen through .transpose(1, 2), say) as
    long as d is contiguous; ``out`` may be strided the same way.  ``mask``
    is an fp32 CUDA tensor addressed with ``mask_strides`` (elements).
    ``fp32_tc`` selects, for fp32 tensors, the tensor-core path with three
    TF32 products per matrix product (FA_DTYPE_F32_TC) instead of the SIMT
    one (FA_DTYPE_F32)."""
    import torch
    B, Hq, Tq, d = q.shape
    Hkv, Tk = k.shape[1], k.shape[2]
    _check_tensors(q.device, k=k, v=v, out=out, lse_out=lse_out, sinks=sinks, mask=mask)
    _check_f32("sinks", sinks, Hq)
    _check_f32("mask", mask)
    if isinstance(sinks, torch.Tensor) and not sinks.is_contiguous():
        raise ValueError("sinks must be contiguous [Hq]")
    if q.dtype == torch.float32:
        dt = FA_DTYPE_F32_TC if fp32_tc else FA_DTYPE_F32
    elif q.dtype == torch.bfloat16:
        dt = FA_DTYPE_BF16
    elif q.dtype == torch.float8_e4m3fn:
        dt = FA_DTYPE_FP8_E4M3
    else:
        raise TypeError(f"unsupported dtype {q.dtype}")
    for name, t in (("q", q), ("k", k), ("v", v)) + ((("out", out),) if out is not None else ()):
        if t.dim() != 4 or (t.shape[3] > 1 and t.stride(3) != 1):
            raise ValueError(f"{name} must be 4-D with its last dimension contiguous")
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k and v must share a dtype")
    o_dtype = torch.bfloat16 if dt == FA_DTYPE_FP8_E4M3 else q.dtype
    if out is not None and out.dtype != o_dtype:
        raise TypeError(f"out must be {o_dtype}")
    if lse_out is not None and (not lse_out.is_contiguous() or lse_out.dtype != torch.float32 or
                                lse_out.numel() < B * Hq * Tq):
        raise ValueError("lse_out must be a contiguous float32 [B, Hq, Tq]")
    with torch.cuda.device(q.device):  # the C call launches on the current device
        o = out if out is not None else torch.empty((B, Hq, Tq, d), dtype=o_dtype, device=q.device)
        lse = lse_out if lse_out is not None else (
            torch.empty((B, Hq, Tq), dtype=torch.float32, device=q.device) if with_lse else None)
        sc = (1.0 / d ** 0.5) if scale is None else scale
        fa_fwd_strided(q, k, v, o, lse, B, Hq, Hkv, Tq, Tk, d, q.stride()[:3], k.stride()[:3], v.stride()[:3],
                       o.stride()[:3], sc, q_offset, causal, window, sinks, mask, *mask_strides, dt, stream)
    return o, lse


def fa_fwd_paged(q, k_cache, v_cache, o, lse, B, Hq, Hkv, Tq, d, seq_lens, max_seq_len, block_table, max_blocks,
                 page_size, num_pages, scale, causal, window, sinks, dtype, stream=None, *, check=True) -> int:
    """Call the paged-cache C entry point; raises FaError on a non-OK status
    when ``check``."""
    lib = load()
    st = lib.fa_fwd_paged(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(o), _ptr(lse), int(B), int(Hq), int(Hkv),
                          int(Tq), int(d), _ptr(seq_lens), int(max_seq_len), _ptr(block_table), int(max_blocks),
                          int(page_size), int(num_pages), float(scale), int(bool(causal)), int(window), _ptr(sinks),
                          int(dtype), _stream(stream))
    if check and st != FA_OK:
        raise FaError(st, lib.fa_last_error().decode())
    return st


def paged_attention(q, k_cache, v_cache, block_table, seq_lens, max_seq_len, *, scale=None, causal=True, window=0,
                    sinks=None, stream=None):
    """Decode step on paged caches: q [B, Hq, Tq, d] bf16, k_cache/v_cache
    [num_pages, page_size, Hkv, d] bf16, block_table [B, max_blocks] int32,
    seq_lens [B] int32 (CUDA tensors).  Returns o [B, Hq, Tq, d], lse."""
    import torch
    B, Hq, Tq, d = q.shape
    num_pages, page_size, Hkv, _ = k_cache.shape
    _check_tensors(q.device, k_cache=k_cache, v_cache=v_cache, block_table=block_table, seq_lens=seq_lens,
                   sinks=sinks)
    _check_f32("sinks", sinks, Hq)
    for name, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache), ("block_table", block_table),
                    ("seq_lens", seq_lens)):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if block_table.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise TypeError("block_table and seq_lens must be int32")
    if isinstance(sinks, torch.Tensor) and not sinks.is_contiguous():
        raise ValueError("sinks must be contiguous [Hq]")
    with torch.cuda.device(q.device):  # the C call launches on the current device
        o = torch.empty_like(q)
        lse = torch.empty((B, Hq, Tq), dtype=torch.float32, device=q.device)
        sc = (1.0 / d ** 0.5) if scale is None else scale
        fa_fwd_paged(q, k_cache, v_cache, o, lse, B, Hq, Hkv, Tq, d, seq_lens, max_seq_len, block_table,
                     block_table.shape[1], page_size, num_pages, sc, causal, window, sinks, FA_DTYPE_BF16, stream)
    return o, lse


def fa_fwd_varlen(q, k, v, o, lse, B, Hq, Hkv, d, cu_seqlens_q, cu_seqlens_k, total_q, total_k, max_seqlen_q,
                  max_seqlen_k, q_strides, k_strides, v_strides, o_strides, scale, causal, window, sinks, dtype,
                  stream=None, *, check=True) -> int:
    """Call the variable-length C entry point (each *_strides = (head, row)
    in elements); raises FaError on a non-OK status when ``check``."""
    lib = load()
    st = lib.fa_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), int(B), int(Hq), int(Hkv), int(d),
                           _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), int(total_q), int(total_k), int(max_seqlen_q),
                           int(max_seqlen_k), *[int(x) for x in (*q_strides, *k_strides, *v_strides, *o_strides)],
                           float(scale), int(bool(causal)), int(window), _ptr(sinks), int(dtype), _stream(stream))
    if check and st != FA_OK:
        raise FaError(st, lib.fa_last_error().decode())
    return st


def varlen_attention(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k, *, scale=None, causal=True,
                     window=0, sinks=None, stream=None):
    """Packed sequences: q [total_q, Hq, d], k/v [total_k, Hkv, d] (fp32,
    bf16 or float8_e4m3fn, d contiguous), cu_seqlens_* int32 [B+1] CUDA
    tensors.  Returns o [total_q, Hq, d] (q's dtype; bf16 for e4m3) and lse
    [Hq, total_q]."""
    import torch
    total_q, Hq, d = q.shape
    total_k, Hkv = k.shape[0], k.shape[1]
    B = cu_seqlens_q.numel() - 1
    _check_tensors(q.device, k=k, v=v, cu_seqlens_q=cu_seqlens_q, cu_seqlens_k=cu_seqlens_k, sinks=sinks)
    _check_f32("sinks", sinks, Hq)
    if isinstance(sinks, torch.Tensor) and not sinks.is_contiguous():
        raise ValueError("sinks must be contiguous [Hq]")
    if cu_seqlens_k.numel() != B + 1:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must both hold B + 1 offsets")
    codes = {torch.float32: FA_DTYPE_F32, torch.bfloat16: FA_DTYPE_BF16, torch.float8_e4m3fn: FA_DTYPE_FP8_E4M3}
    if q.dtype not in codes or k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k and v must share a dtype: fp32, bf16 or float8_e4m3fn")
    dt = codes[q.dtype]
    if cu_seqlens_q.dtype != torch.int32 or cu_seqlens_k.dtype != torch.int32:
        raise TypeError("cu_seqlens must be int32")
    with torch.cuda.device(q.device):  # the C call launches on the current device
        o = torch.empty((total_q, Hq, d), dtype=torch.bfloat16 if dt == FA_DTYPE_FP8_E4M3 else q.dtype,
                        device=q.device)
        lse = torch.empty((Hq, total_q), dtype=torch.float32, device=q.device)
        sc = (1.0 / d ** 0.5) if scale is None else scale
        fa_fwd_varlen(q, k, v, o, lse, B, Hq, Hkv, d, cu_seqlens_q, cu_seqlens_k, total_q, total_k, max_seqlen_q,
                      max_seqlen_k, (q.stride(1), q.stride(0)), (k.stride(1), k.stride(0)),
                      (v.stride(1), v.stride(0)), (o.stride(1), o.stride(0)), sc, causal, window, sinks, dt, stream)
    return o, lse
