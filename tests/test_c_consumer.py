"""The C ABI from plain C: include/fa.h compiles as C99 (and with -Wall
-Wextra -Werror), and a C program linked against libfa.so gets the version
and the argument errors, which are returned before any launch (no GPU
needed)."""
from __future__ import annotations

import shutil
import subprocess
from pathlib import Path

import pytest

import exact_tiled_attention_flashattention_gb300 as fa

_ROOT = Path(__file__).resolve().parents[1]

_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "fa.h"

int main(void) {
    int bad = 0;
    if (fa_version() < 100) { printf("version %d\n", fa_version()); ++bad; }
    /* negative size */
    fa_status st = fa_fwd(NULL, NULL, NULL, NULL, NULL, 1, 2, 1, -5, 8, 64, 0.125f, 0, 1, 0, NULL, NULL, 0, 0, 0, 0,
                          FA_DTYPE_BF16, NULL);
    if (st != FA_EINVAL || strlen(fa_last_error()) == 0) { printf("negative size: %d\n", (int)st); ++bad; }
    /* 3 query heads on 2 KV heads */
    st = fa_fwd(NULL, NULL, NULL, NULL, NULL, 1, 3, 2, 8, 8, 64, 0.125f, 0, 1, 0, NULL, NULL, 0, 0, 0, 0,
                FA_DTYPE_F32, NULL);
    if (st != FA_ESHAPE) { printf("shape: %d\n", (int)st); ++bad; }
    /* unknown dtype */
    st = fa_fwd(NULL, NULL, NULL, NULL, NULL, 1, 2, 1, 8, 8, 64, 0.125f, 0, 1, 0, NULL, NULL, 0, 0, 0, 0, 7, NULL);
    if (st != FA_EINVAL) { printf("dtype: %d\n", (int)st); ++bad; }
    /* an empty problem is a no-op */
    st = fa_fwd(NULL, NULL, NULL, NULL, NULL, 0, 2, 1, 8, 8, 64, 0.125f, 0, 1, 0, NULL, NULL, 0, 0, 0, 0,
                FA_DTYPE_BF16, NULL);
    if (st != FA_OK || fa_last_error()[0] != '\0') { printf("empty: %d\n", (int)st); ++bad; }
    /* paged: bf16 only */
    st = fa_fwd_paged(NULL, NULL, NULL, NULL, NULL, 1, 2, 1, 1, 64, NULL, 0, NULL, 0, 16, 1, 0.125f, 1, 0, NULL,
                      FA_DTYPE_F32, NULL);
    if (st == FA_OK) { printf("paged fp32 accepted\n"); ++bad; }
    printf("failures %d\n", bad);
    return bad;
}
"""


def _gcc():
    g = shutil.which("gcc")
    if g is None:
        pytest.skip("no C compiler")
    return g


def test_header_compiles_as_c99(tmp_path):
    src = tmp_path / "h.c"
    src.write_text('#include "fa.h"\nint f(void) { return (int)FA_DTYPE_FP8_E4M3 + (int)FA_ETIMEOUT; }\n')
    subprocess.run([_gcc(), "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", f"-I{_ROOT / 'include'}", "-c",
                    str(src), "-o", str(tmp_path / "h.o")], check=True)


def test_c_program_links_and_gets_the_errors(tmp_path):
    lib = fa.library_path()
    if not lib.exists():
        pytest.skip("libfa.so not built")
    src = tmp_path / "prog.c"
    src.write_text(_PROGRAM)
    exe = tmp_path / "prog"
    subprocess.run([_gcc(), "-std=c99", "-Wall", "-Werror", f"-I{_ROOT / 'include'}", str(src), str(lib),
                    f"-Wl,-rpath,{lib.parent}", "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "failures 0" in r.stdout
