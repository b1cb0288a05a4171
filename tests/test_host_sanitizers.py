"""Host code under the compiler's sanitizers (CPU only, no GPU involved).

compute-sanitizer is not available for the kernels, so the host-side code is
checked the way "FlashAttention forward in C" checks its C kernel (ASan,
UBSan and TSan builds):

* the argument validation of the C ABI (``csrc/fa_api.cu``, host code only)
  is compiled with g++ under AddressSanitizer and UndefinedBehaviorSanitizer,
  with stand-in launchers that only record the parameters they receive, and
  driven through every entry point with a battery of extreme arguments
  (sizes and strides near 0, 2^30, 2^31, 2^40, 2^62 and INT64_MAX, negative
  values, NULL and misaligned pointers, unknown dtypes, non-finite scales).
  No signed overflow or out-of-bounds access may occur, every call must
  return a status of the ABI, and no launcher may be reached by a call that
  returned an error;
* the float64 oracle is run on small problems of every flag combination,
  with masks, sinks, row subsets and several threads, under ASan + UBSan and
  under ThreadSanitizer.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from pathlib import Path

import pytest

_ROOT = Path(__file__).resolve().parents[1]
_CSRC = _ROOT / "exact_tiled_attention_flashattention_gb300" / "csrc"
_ORACLE = _ROOT / "oracle" / "fa_oracle.c"

_STUBS = r"""
#include "fa_internal.h"
namespace fa {
Params g_last;
int g_calls = 0;
long g_bad_grids = 0;
// Every accepted call must give a grid the kernels can index with 31-bit
// block numbers: query tiles of `rows` rows of every (batch, head).
static void grid_ok(const Params &P, long long rows) {
    const long long tiles = ((long long)P.Tq + rows - 1) / rows;
    if (P.B < 0 || P.Hq < 0 || P.Tq < 0 || tiles * P.B * P.Hq > 0x7fffffffll) ++g_bad_grids;
}
#define FA_STUB(name, rows) \
    cudaError_t name(const Params &P, cudaStream_t) { g_last = P; ++g_calls; grid_ok(P, rows); return cudaSuccess; }
FA_STUB(launch_f32, 64)
FA_STUB(launch_f32_tc, 128)
FA_STUB(launch_bf16, 128)
FA_STUB(launch_fp8, 128)
FA_STUB(launch_fp8_varlen, 128)
FA_STUB(launch_bf16_paged, 128)
FA_STUB(launch_bf16_varlen, 128)
FA_STUB(launch_f32_varlen, 64)
cudaError_t launch_bf16_splitkv(const Params &P, void *, cudaStream_t) {
    g_last = P; ++g_calls; grid_ok(P, 128); return cudaSuccess;
}
cudaError_t launch_bf16_splitkv_noalloc(const Params &P, cudaStream_t) {
    g_last = P; ++g_calls; grid_ok(P, 128); return cudaSuccess;
}
// The sizing rule of the real launcher with a fixed SM count of 152.
size_t splitkv_workspace_bytes(int B, int Hkv, int group, int Tq, int d) {
    if ((long long)group * Tq > 128 || B <= 0 || Hkv <= 0 || Tq <= 0 || d <= 0) return 0;
    const long long units = (long long)B * Hkv;
    if (units > 0x7fffffffll) { ++g_bad_grids; return 0; }
    long long S = 152 / units;
    S = S < 1 ? 1 : (S > 64 ? 64 : S);
    const long long blk = ((long long)group * Tq * ((d <= 64 ? 64 : 128) + 2) + 3) / 4 * 4;  // 16-byte blocks
    return (size_t)((units * 4 + 255) / 256 * 256) + (size_t)units * S * blk * 4;
}
cudaError_t bf16_watchdog(cudaStream_t, unsigned int *f) { *f = 0; return cudaSuccess; }
cudaError_t f32tc_watchdog(cudaStream_t, unsigned int *f) { *f = 0; return cudaSuccess; }
cudaError_t bf16_set_drop_arrive(int) { return cudaSuccess; }
cudaError_t f32tc_set_drop_arrive(int) { return cudaSuccess; }
}  // namespace fa
"""

_API_DRIVER = r"""
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <limits>
#include "fa.h"
#include "fa_internal.h"
namespace fa { extern Params g_last; extern int g_calls; extern long g_bad_grids; }

static uint64_t state = 0x243f6a8885a308d3ull;
static uint64_t next() {  // xorshift64*
    state ^= state >> 12; state ^= state << 25; state ^= state >> 27;
    return state * 0x2545f4914f6cdd1dull;
}
static const int64_t kI64Max = std::numeric_limits<int64_t>::max();
static const int64_t kI64Min = std::numeric_limits<int64_t>::min();
static const int64_t kVals[] = {0, 1, 2, 3, 4, 7, 8, 16, 63, 64, 96, 127, 128, 129, 256, 1000, 4096,
                                (1ll << 24) - 1, 1ll << 24, (1ll << 30) - 1, 1ll << 30, (1ll << 31) - 1,
                                1ll << 31, 1ll << 32, 1ll << 40, 1ll << 62, kI64Max, -1, -8, -(1ll << 31),
                                kI64Min};
static int64_t pick() {
    const uint64_t r = next();
    if (r % 4 == 0) return (int64_t)(next() % 300);  // small values, the common case
    return kVals[r % (sizeof kVals / sizeof kVals[0])];
}
static const void *ptr() {
    static const uintptr_t p[] = {0, 0x100000, 0x100000, 0x100010, 0x100008, 0x100001};
    return reinterpret_cast<const void *>(p[next() % 6]);
}
static float scale() {
    static const float s[] = {0.125f, 0.125f, 1.f, 0.f, -0.5f, INFINITY, NAN};
    return s[next() % 7];
}
static long bad = 0;
static void check(const char *entry, fa_status st, int calls_before) {
    if ((int)st < 0 || (int)st > 5) {
        if (bad++ < 5) std::printf("%s: status %d outside the ABI\n", entry, (int)st);
    }
    if (st != FA_OK && fa::g_calls != calls_before) {
        if (bad++ < 5) std::printf("%s: launched although it returned %d\n", entry, (int)st);
    }
    if (st != FA_OK && fa_last_error()[0] == '\0') {
        if (bad++ < 5) std::printf("%s: status %d without a message\n", entry, (int)st);
    }
}

int main() {
    void *const out = reinterpret_cast<void *>(0x200000);
    float *const lse = reinterpret_cast<float *>(0x300000);
    long n = 0;
    for (int it = 0; it < 60000; ++it) {
        const int dtype = (int)(next() % 6) - 1;  // -1 .. 4: two unknown codes
        int c = fa::g_calls;
        fa_status st = fa_fwd(ptr(), ptr(), ptr(), out, (next() & 1) ? lse : nullptr, pick(), pick(), pick(), pick(),
                              pick(), pick(), scale(), pick(), (int)(next() & 1), pick(),
                              (next() & 1) ? (const float *)ptr() : nullptr, (next() & 1) ? (const float *)ptr() : nullptr,
                              pick(), pick(), pick(), pick(), dtype, nullptr);
        check("fa_fwd", st, c);
        c = fa::g_calls;
        st = fa_fwd_strided(ptr(), ptr(), ptr(), out, lse, pick(), pick(), pick(), pick(), pick(), pick(), pick(),
                            pick(), pick(), pick(), pick(), pick(), pick(), pick(), pick(), pick(), pick(), pick(),
                            scale(), pick(), (int)(next() & 1), pick(), nullptr, nullptr, 0, 0, 0, 0, dtype, nullptr);
        check("fa_fwd_strided", st, c);
        c = fa::g_calls;
        st = fa_fwd_paged(ptr(), ptr(), ptr(), out, lse, pick(), pick(), pick(), pick(), pick(),
                          (const int32_t *)ptr(), pick(), (const int32_t *)ptr(), pick(), pick(), pick(), scale(),
                          (int)(next() & 1), pick(), nullptr, dtype, nullptr);
        check("fa_fwd_paged", st, c);
        c = fa::g_calls;
        st = fa_fwd_varlen(ptr(), ptr(), ptr(), out, lse, pick(), pick(), pick(), pick(), (const int32_t *)ptr(),
                           (const int32_t *)ptr(), pick(), pick(), pick(), pick(), pick(), pick(), pick(), pick(),
                           pick(), pick(), pick(), pick(), scale(), (int)(next() & 1), pick(), nullptr, dtype,
                           nullptr);
        check("fa_fwd_varlen", st, c);
        c = fa::g_calls;
        st = fa_fwd_splitkv(ptr(), ptr(), ptr(), out, lse, pick(), pick(), pick(), pick(), pick(), pick(), scale(),
                            pick(), (int)(next() & 1), pick(), nullptr, nullptr, 0, 0, 0, 0,
                            (next() & 1) ? (void *)ptr() : nullptr, (size_t)pick(), dtype, nullptr);
        check("fa_fwd_splitkv", st, c);
        c = fa::g_calls;
        st = fa_fwd_splitkv_noalloc(ptr(), ptr(), ptr(), out, lse, pick(), pick(), pick(), pick(), pick(), pick(),
                                    scale(), pick(), (int)(next() & 1), pick(), nullptr, nullptr, 0, 0, 0, 0, dtype,
                                    nullptr);
        check("fa_fwd_splitkv_noalloc", st, c);
        size_t ws = 0;
        st = fa_splitkv_workspace_bytes(pick(), pick(), pick(), pick(), pick(), dtype, (next() & 7) ? &ws : nullptr);
        check("fa_splitkv_workspace_bytes", st, fa::g_calls);
        n += 6;
    }
    // Arguments that pass the earlier checks and reach the products of the
    // later ones: a page size near 2^62 with no pages, a varlen batch whose
    // head count only the output strides bound.
    const void *a = reinterpret_cast<const void *>(0x100000);
    const int32_t *ia = reinterpret_cast<const int32_t *>(0x100000);
    for (int64_t mb : {int64_t(4), int64_t(1) << 20, kI64Max}) {
        int c = fa::g_calls;
        fa_status st = fa_fwd_paged(a, a, a, out, lse, 1, 2, 1, 1, 64, ia, 100, ia, mb, int64_t(1) << 62, 0, 0.125f,
                                    1, 0, nullptr, FA_DTYPE_BF16, nullptr);
        check("fa_fwd_paged (huge pages)", st, c);
        if (st == FA_OK && bad++ < 5) std::printf("paged call with no pages accepted\n");
    }
    for (int64_t B : {int64_t(2), int64_t(1) << 20}) {
        const int64_t Hq = int64_t(1) << 50;
        int c = fa::g_calls;
        fa_status st = fa_fwd_varlen(a, a, a, out, lse, B, Hq, Hq, 64, ia, ia, 10, 10, 10, 10, 0, 64, 0, 64, 0, 64,
                                     64, 64 * Hq, 0.125f, 1, 0, nullptr, FA_DTYPE_BF16, nullptr);
        check("fa_fwd_varlen (huge head count)", st, c);
        if (st == FA_OK && bad++ < 5) std::printf("varlen call with 2^50 heads accepted\n");
    }
    // A valid call reaches its launcher with the contiguous strides.
    int c = fa::g_calls;
    fa_status st = fa_fwd(a, a, a, out, lse, 2, 16, 8, 511, 511, 128, 0.088f, 0, 1, 0, nullptr, nullptr, 0, 0, 0, 0,
                          FA_DTYPE_BF16, nullptr);
    if (st != FA_OK || fa::g_calls != c + 1 || fa::g_last.q_sb != 16ll * 511 * 128 || fa::g_last.k_sh != 511ll * 128 ||
        fa::g_last.group != 2 || fa::g_last.Tq != 511) {
        std::printf("valid call: status %d, %s\n", (int)st, fa_last_error());
        ++bad;
    }
    // Split-KV: a decode step needs the size the query reports; one byte less
    // is refused before any launch, the exact size reaches the launcher.
    {
        size_t need = 0;
        fa_status st = fa_splitkv_workspace_bytes(2, 16, 8, 1, 128, FA_DTYPE_BF16, &need);
        void *ws = reinterpret_cast<void *>(0x400000);
        int c = fa::g_calls;
        fa_status st2 = fa_fwd_splitkv(a, a, a, out, lse, 2, 16, 8, 1, 4096, 128, 0.088f, 4095, 1, 0, nullptr, nullptr,
                                       0, 0, 0, 0, ws, need - 1, FA_DTYPE_BF16, nullptr);
        check("fa_fwd_splitkv (short workspace)", st2, c);
        if (st != FA_OK || need == 0 || st2 != FA_EINVAL) {
            std::printf("split-KV sizing: %d %zu %d\n", (int)st, need, (int)st2);
            ++bad;
        }
        c = fa::g_calls;
        st2 = fa_fwd_splitkv(a, a, a, out, lse, 2, 16, 8, 1, 4096, 128, 0.088f, 4095, 1, 0, nullptr, nullptr, 0, 0, 0,
                             0, ws, need, FA_DTYPE_BF16, nullptr);
        if (st2 != FA_OK || fa::g_calls != c + 1 || fa::g_last.Tk != 4096 || fa::g_last.group != 2) {
            std::printf("split-KV valid call: status %d, %s\n", (int)st2, fa_last_error());
            ++bad;
        }
    }
    // The static-scratch variant: a call whose workspace exceeds the array is
    // refused before any launch; a decode step within it is launched.
    {
        int c = fa::g_calls;
        fa_status st = fa_fwd_splitkv_noalloc(a, a, a, out, lse, 200, 128, 8, 8, 4096, 128, 0.088f, 4088, 1, 0,
                                              nullptr, nullptr, 0, 0, 0, 0, FA_DTYPE_BF16, nullptr);
        check("fa_fwd_splitkv_noalloc (oversize)", st, c);
        if (st != FA_EUNSUPPORTED || std::strstr(fa_last_error(), "scratch") == nullptr) {
            std::printf("oversize no-alloc call: status %d, %s\n", (int)st, fa_last_error());
            ++bad;
        }
        c = fa::g_calls;
        st = fa_fwd_splitkv_noalloc(a, a, a, out, lse, 1, 16, 8, 1, 32768, 128, 0.088f, 32767, 1, 0, nullptr, nullptr,
                                    0, 0, 0, 0, FA_DTYPE_BF16, nullptr);
        if (st != FA_OK || fa::g_calls != c + 1 || fa::g_last.Tk != 32768) {
            std::printf("no-alloc decode step: status %d, %s\n", (int)st, fa_last_error());
            ++bad;
        }
    }
    // fp32 on the SIMT cores: 64-row tiles, so 2^31 tiles come sooner.
    {
        int c = fa::g_calls;
        // B * Hq = 2^23 heads of 2^14 rows: 2^31 tiles of 64 rows; q, k and v
        // broadcast (stride 0), o distinct rows of d = 2
        fa_status st = fa_fwd_strided(a, a, a, out, lse, 1 << 19, 1 << 4, 1 << 4, 1 << 14, 1, 2, 0, 0, 0, 0, 0, 0, 0, 0,
                                      0, int64_t(1) << 19, int64_t(1) << 15, 2, 0.125f, 0, 0, 0, nullptr, nullptr, 0,
                                      0, 0, 0, FA_DTYPE_F32, nullptr);
        check("fa_fwd_strided (2^31 fp32 tiles)", st, c);
        if (st == FA_OK && bad++ < 5) std::printf("fp32 call with 2^31 query tiles accepted\n");
    }
    if (fa::g_bad_grids != 0) {
        std::printf("%ld accepted calls with a grid of 2^31 tiles or more\n", fa::g_bad_grids);
        ++bad;
    }
    std::printf("calls %ld, launched %d, failures %ld\n", n + 1, fa::g_calls, bad);
    return bad == 0 ? 0 : 1;
}
"""

_ORACLE_DRIVER = r"""
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

int fa_oracle_f64(const double *q, const double *k, const double *v, double *o, double *lse,
                  int64_t B, int64_t Hq, int64_t Hkv, int64_t Tq, int64_t Tk, int64_t D,
                  double scale, int64_t q_offset, int causal, int64_t window,
                  const double *sinks, const double *mask, int64_t msb, int64_t msh,
                  int64_t msq, int64_t msk, const int64_t *rows, int64_t nrows, int nthreads);

static uint64_t state = 0x13198a2e03707344ull;
static uint64_t next(void) {
    state ^= state >> 12; state ^= state << 25; state ^= state >> 27;
    return state * 0x2545f4914f6cdd1dull;
}
static double *randn(int64_t n) {
    double *p = (double *)malloc((size_t)(n > 0 ? n : 1) * sizeof(double));
    for (int64_t i = 0; i < n; ++i) p[i] = (double)(next() % 2001) / 1000.0 - 1.0;
    return p;
}

int main(void) {
    static const int64_t T[] = {0, 1, 2, 5, 17};
    long bad = 0, runs = 0;
    for (int it = 0; it < ITERS; ++it) {
        const int64_t B = (int64_t)(next() % 3), Hkv = 1 + (int64_t)(next() % 2), Hq = Hkv * (1 + (int64_t)(next() % 3));
        const int64_t Tq = T[next() % 5], Tk = T[next() % 5], D = 1 + (int64_t)(next() % 8);
        const int64_t q_offset = (int64_t)(next() % 3) * 7, window = (int64_t)(next() % 4);
        const int causal = (int)(next() & 1), mode = (int)(next() % 3), nthreads = 1 + (int)(next() % 3);
        double *q = randn(B * Hq * Tq * D), *k = randn(B * Hkv * Tk * D), *v = randn(B * Hkv * Tk * D);
        double *sinks = (next() & 1) ? randn(Hq) : NULL;
        /* mask: none, broadcast [Tq, Tk] (strides 0, 0, Tk, 1) or full [B, Hq, Tq, Tk] */
        double *mask = NULL;
        int64_t msb = 0, msh = 0, msq = 0, msk = 0;
        if (mode == 1) { mask = randn(Tq * Tk); msq = Tk; msk = 1; }
        if (mode == 2) { mask = randn(B * Hq * Tq * Tk); msb = Hq * Tq * Tk; msh = Tq * Tk; msq = Tk; msk = 1; }
        if (mask) for (int64_t i = 0; i < (mode == 1 ? Tq * Tk : B * Hq * Tq * Tk); ++i)
            if (next() % 5 == 0) mask[i] = -INFINITY;
        int64_t rows[4], nrows = 0;
        const int subset = Tq > 0 && (next() & 1);
        if (subset) { nrows = 1 + (int64_t)(next() % 4); for (int64_t r = 0; r < nrows; ++r) rows[r] = (int64_t)(next() % (uint64_t)Tq); }
        const int64_t R = subset ? nrows : Tq;
        double *o = randn(B * Hq * R * D), *lse = randn(B * Hq * R);
        const int st = fa_oracle_f64(q, k, v, o, lse, B, Hq, Hkv, Tq, Tk, D, 0.3, q_offset, causal, window, sinks, mask,
                                     msb, msh, msq, msk, subset ? rows : NULL, nrows, nthreads);
        if (st != 0) { if (bad++ < 5) printf("valid problem rejected: %d\n", st); }
        for (int64_t i = 0; i < B * Hq * R; ++i)
            if (isnan(lse[i])) { if (bad++ < 5) printf("NaN lse\n"); break; }
        ++runs;
        /* invalid arguments are rejected before anything is written */
        if (fa_oracle_f64(q, k, v, o, lse, B, 3, 2, Tq, Tk, D, 0.3, 0, 0, 0, NULL, NULL, 0, 0, 0, 0, NULL, 0, 1) != 2)
            if (bad++ < 5) printf("3 heads on 2 KV heads accepted\n");
        if (Tq > 0) {
            int64_t badrow = Tq;
            if (fa_oracle_f64(q, k, v, o, lse, B, Hq, Hkv, Tq, Tk, D, 0.3, 0, 0, 0, NULL, NULL, 0, 0, 0, 0, &badrow, 1,
                              1) == 0)
                if (bad++ < 5) printf("row out of range accepted\n");
        }
        free(q); free(k); free(v); free(o); free(lse); free(sinks); free(mask);
    }
    printf("runs %ld, failures %ld\n", runs, bad);
    return bad == 0 ? 0 : 1;
}
"""


def _compiler(name):
    c = shutil.which(name)
    if c is None:
        pytest.skip(f"no {name}")
    return c


def _cuda_include():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    inc = Path(nvcc).resolve().parent.parent / "include"
    if not (inc / "cuda_runtime.h").exists():
        pytest.skip("CUDA headers not found")
    return inc


def _run(cmd, exe, timeout=600):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0 and "sanitizer" in (r.stderr + r.stdout).lower() and "cannot" in r.stderr.lower():
        pytest.skip("sanitizer runtime unavailable: " + r.stderr[-200:])
    assert r.returncode == 0, r.stdout + r.stderr
    env = dict(os.environ, ASAN_OPTIONS="detect_leaks=1:abort_on_error=0", UBSAN_OPTIONS="print_stacktrace=1",
               TSAN_OPTIONS="halt_on_error=1")
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=timeout, env=env)
    out = r.stdout + r.stderr
    assert r.returncode == 0 and "runtime error" not in out and "ERROR:" not in out and "WARNING:" not in out, out
    assert "failures 0" in r.stdout, out
    return r.stdout


def test_abi_validation_under_asan_ubsan(tmp_path):
    gxx = _compiler("g++")
    inc = _cuda_include()
    (tmp_path / "stubs.cpp").write_text(_STUBS)
    (tmp_path / "driver.cpp").write_text(_API_DRIVER)
    libdir = inc.parent / "lib64"
    exe = tmp_path / "api_san"
    cmd = [gxx, "-std=c++17", "-O1", "-g", "-fsanitize=address,undefined", "-fno-sanitize-recover=all",
           "-fno-omit-frame-pointer", f"-I{_CSRC}", f"-I{_ROOT / 'include'}", f"-I{inc}",
           "-x", "c++", str(_CSRC / "fa_api.cu"), "-x", "none", str(tmp_path / "stubs.cpp"),
           str(tmp_path / "driver.cpp"), f"-L{libdir}", "-lcudart", f"-Wl,-rpath,{libdir}", "-o", str(exe)]
    out = _run(cmd, exe)
    assert "launched" in out


@pytest.mark.parametrize("san", ["address,undefined", "thread"])
def test_oracle_under_sanitizers(tmp_path, san):
    gcc = _compiler("gcc")
    (tmp_path / "driver.c").write_text(_ORACLE_DRIVER)
    exe = tmp_path / "oracle_san"
    iters = 3000 if san == "thread" else 6000
    cmd = [gcc, "-std=c11", "-O1", "-g", f"-fsanitize={san}", "-fno-omit-frame-pointer", f"-DITERS={iters}",
           "-pthread", str(_ORACLE), str(tmp_path / "driver.c"), "-lm", "-o", str(exe)]
    if san != "thread":
        cmd.insert(4, "-fno-sanitize-recover=all")
    _run(cmd, exe)
