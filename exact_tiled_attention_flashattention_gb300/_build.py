"""Build of libfa.so: the CUDA kernels and the C ABI, compiled for sm_103a.

Each translation unit is compiled in parallel with nvcc, then linked into one
shared library in the package directory (in-tree, git-ignored).  Nothing here
runs at import time; ``build()`` is called by the repository's build entry.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

PKG = Path(__file__).resolve().parent
CSRC = PKG / "csrc"
INCLUDE = PKG.parent / "include"
LIB = PKG / "libfa.so"
OBJ_DIR = PKG / "_build"

SOURCES = ["fa_api.cu", "fa_fwd_f32.cu", "fa_fwd_bf16.cu", "fa_fwd_f32tc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not Path(cand).exists():
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libfa.so")
    return cand


def _cuda_lib_dir(nvcc: str) -> Path:
    return Path(nvcc).resolve().parent.parent / "lib64"


def build(verbose: bool = False, force: bool = False) -> Path:
    """Compile every kernel and link ``libfa.so``; returns its path."""
    nvcc = _nvcc()
    OBJ_DIR.mkdir(exist_ok=True)
    headers = list(CSRC.glob("*.h")) + list(CSRC.glob("*.cuh")) + list(INCLUDE.glob("*.h"))
    newest_header = max((h.stat().st_mtime for h in headers), default=0.0)
    common = [nvcc, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", str(INCLUDE),
              "--expt-relaxed-constexpr"]
    if verbose:
        common += ["-Xptxas", "-v"]

    def compile_one(src: str) -> Path:
        s = CSRC / src
        o = OBJ_DIR / (Path(src).stem + ".o")
        if not force and o.exists() and o.stat().st_mtime >= max(s.stat().st_mtime, newest_header):
            return o
        cmd = common + ["-c", str(s), "-o", str(o)]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr)
        return o

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    if force or not LIB.exists() or LIB.stat().st_mtime < max(o.stat().st_mtime for o in objs):
        tmp = LIB.with_name(LIB.name + f".tmp{os.getpid()}")
        libdir = _cuda_lib_dir(nvcc)
        cmd = [nvcc, *ARCH, "-shared", "-o", str(tmp), *map(str, objs), "-cudart", "shared",
               "-Xlinker", f"-rpath,{libdir}"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link of libfa.so failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv))
