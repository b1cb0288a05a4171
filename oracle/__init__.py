"""Float64 CPU oracle for exact attention -- test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA path never imports it and the
two share no code; both only read the seeded inputs made by ``workloads``.

The arithmetic lives in ``fa_oracle.c`` (plain C, float64, one query row at a
time).  It states the definition of "FlashAttention forward in C", section 2.1,
with the additive strided mask of "Fused attention and softmax: fast and
exact" ("What is computed").  This module only builds the C file with gcc and
marshals numpy arrays to it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "fa_oracle.c"
_LIB = _HERE / "libfa_oracle.so"

_c_i64 = ctypes.c_int64
_c_dp = ctypes.POINTER(ctypes.c_double)
_c_ip = ctypes.POINTER(ctypes.c_int64)


def build(mutant: int = 0, out: Path | None = None) -> Path:
    """Compile the oracle with gcc.  ``mutant`` plants one known mistake
    (for the mutant tests); 0 builds the real oracle."""
    out = Path(out) if out is not None else _LIB
    if mutant == 0 and out == _LIB and out.exists() and out.stat().st_mtime >= _SRC.stat().st_mtime:
        return out
    out.parent.mkdir(parents=True, exist_ok=True)
    tmp = out.with_name(out.name + f".tmp{os.getpid()}")
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", f"-DORACLE_MUTANT={int(mutant)}",
           str(_SRC), "-o", str(tmp), "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


class Oracle:
    """One loaded build of the oracle library (the real one or a mutant)."""

    def __init__(self, path: Path):
        self.path = Path(path)
        self._lib = ctypes.CDLL(str(self.path))
        f = self._lib.fa_oracle_f64
        f.restype = ctypes.c_int
        f.argtypes = [_c_dp, _c_dp, _c_dp, _c_dp, _c_dp,
                      _c_i64, _c_i64, _c_i64, _c_i64, _c_i64, _c_i64,
                      ctypes.c_double, _c_i64, ctypes.c_int, _c_i64,
                      _c_dp, _c_dp, _c_i64, _c_i64, _c_i64, _c_i64,
                      _c_ip, _c_i64, ctypes.c_int]
        self._f = f

    def raw(self, q, k, v, o, lse, B, Hq, Hkv, Tq, Tk, D, scale, q_offset, causal, window,
            sinks, mask, strides, rows, nthreads):
        """Direct call with numpy float64 buffers (or None); returns the status."""
        def dp(a):
            return None if a is None else a.ctypes.data_as(_c_dp)
        rp = None if rows is None else rows.ctypes.data_as(_c_ip)
        nrows = 0 if rows is None else int(rows.size)
        sb, sh, sq, sk = strides
        return self._f(dp(q), dp(k), dp(v), dp(o), dp(lse), B, Hq, Hkv, Tq, Tk, D,
                       float(scale), int(q_offset), int(bool(causal)), int(window),
                       dp(sinks), dp(mask), sb, sh, sq, sk, rp, nrows, int(nthreads))

    def attention(self, q, k, v, scale, *, q_offset=0, causal=False, window=0, sinks=None,
                  mask=None, mask_strides=(0, 0, 0, 0), rows=None, threads=None):
        """o [B,Hq,R,D], lse [B,Hq,R] in float64 (R = len(rows) or Tq).

        q [B,Hq,Tq,D]; k, v [B,Hkv,Tk,D]; sinks [Hq] or None; mask a flat
        buffer indexed with ``mask_strides`` (elements) or None.  Inputs of any
        float dtype are widened to float64 exactly.
        """
        q = np.ascontiguousarray(np.asarray(q, dtype=np.float64))
        k = np.ascontiguousarray(np.asarray(k, dtype=np.float64))
        v = np.ascontiguousarray(np.asarray(v, dtype=np.float64))
        B, Hq, Tq, D = q.shape
        _, Hkv, Tk, _ = k.shape
        if rows is not None:
            rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        R = Tq if rows is None else int(rows.size)
        o = np.zeros((B, Hq, R, D), dtype=np.float64)
        lse = np.zeros((B, Hq, R), dtype=np.float64)
        if sinks is not None:
            sinks = np.ascontiguousarray(np.asarray(sinks, dtype=np.float64))
        if mask is not None:
            mask = np.ascontiguousarray(np.asarray(mask, dtype=np.float64)).reshape(-1)
        nt = threads if threads is not None else (os.cpu_count() or 1)
        st = self.raw(q, k, v, o, lse, B, Hq, Hkv, Tq, Tk, D, scale, q_offset, causal, window,
                      sinks, mask, tuple(int(s) for s in mask_strides), rows, nt)
        if st != 0:
            raise ValueError(f"oracle rejected the arguments (status {st})")
        return o, lse


_default: Oracle | None = None


def get() -> Oracle:
    """The real oracle, built on first use."""
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default


def attention(*args, **kwargs):
    """Shorthand for ``get().attention(...)``."""
    return get().attention(*args, **kwargs)
