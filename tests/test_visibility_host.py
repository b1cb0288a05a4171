"""Host check of the kernels' visible-key interval (csrc/fa_internal.h).

The tensor-core kernels mask each row by the interval [lo, hi) that
``visible_range_tk`` returns, and size each unit's walk over key tiles from
the intervals of its first and last rows.  That function is compiled for the
host as well; here it is compared with the visibility rule of "FlashAttention
forward in C" (section 2.1) applied key by key: j is visible from position p
iff j < Tk, (not causal or j <= p) and (w <= 0 or j > p - w).  Also checked:
the interval moves monotonically with p, so the keys of a 128-row query tile
are exactly the keys from its first row's lo to its last row's hi, which is
the range the kernels walk.  And the bit mask of a thread's interval
among its 64 keys of a tile (``key_bits``), which the kernels test on
boundary tiles, against the interval itself.
"""
from __future__ import annotations

import shutil
import subprocess
from pathlib import Path

import pytest

_ROOT = Path(__file__).resolve().parents[1]
_CSRC = _ROOT / "exact_tiled_attention_flashattention_gb300" / "csrc"

_DRIVER = r"""
#include <cstdint>
#include <cstdio>
#include <cstring>
#include "fa_internal.h"

static uint64_t state = 0x452821e638d01377ull;
static uint64_t next() {
    state ^= state >> 12; state ^= state << 25; state ^= state >> 27;
    return state * 0x2545f4914f6cdd1dull;
}
static bool visible(int64_t j, int64_t p, int64_t Tk, int causal, int64_t w) {
    if (j >= Tk) return false;
    if (causal && j > p) return false;
    if (w > 0 && j <= p - w) return false;
    return true;
}
static long bad = 0, checked = 0;

int main() {
    fa::Params P;
    // Brute force on small sizes: every key of every position.
    for (int causal = 0; causal < 2; ++causal)
        for (int w = -1; w <= 9; ++w)
            for (int64_t Tk = 0; Tk <= 40; ++Tk)
                for (int64_t p = 0; p <= 60; ++p) {
                    std::memset(&P, 0, sizeof P);
                    P.causal = causal;
                    P.window = w;
                    int64_t lo, hi;
                    fa::visible_range_tk(P, Tk, p, lo, hi);
                    ++checked;
                    if (lo < 0 || hi < lo || hi > (Tk > lo ? Tk : lo)) {
                        if (bad++ < 5) std::printf("bad interval [%lld, %lld) Tk=%lld p=%lld\n", (long long)lo, (long long)hi, (long long)Tk, (long long)p);
                    }
                    for (int64_t j = 0; j < Tk + 3; ++j)
                        if (visible(j, p, Tk, causal, w) != (j >= lo && j < hi)) {
                            if (bad++ < 5)
                                std::printf("key %lld: causal=%d w=%d Tk=%lld p=%lld -> [%lld, %lld)\n", (long long)j,
                                            causal, w, (long long)Tk, (long long)p, (long long)lo, (long long)hi);
                        }
                }
    // Large positions and windows: the interval's ends against the rule at
    // and next to them, and monotonicity in p over 128 consecutive rows.
    for (int it = 0; it < 200000; ++it) {
        std::memset(&P, 0, sizeof P);
        P.causal = (int)(next() & 1);
        const uint64_t r = next() % 4;
        P.window = r == 0 ? 0 : (int)(next() % (r == 1 ? 300 : (1u << 31) - 1));
        const int64_t Tk = (int64_t)(next() % (1u << 30));
        const int64_t p0 = (int64_t)(next() % ((1ull << 31) + 200));
        int64_t plo = -1, phi = -1, first_lo = 0, union_hi = 0;
        bool any = false;
        for (int64_t p = p0; p < p0 + 128; ++p) {
            int64_t lo, hi;
            fa::visible_range_tk(P, Tk, p, lo, hi);
            ++checked;
            if (p > p0 && (lo < plo || hi < phi)) {
                if (bad++ < 5) std::printf("not monotonic at p=%lld\n", (long long)p);
            }
            plo = lo;
            phi = hi;
            if (p == p0) first_lo = lo;
            if (hi > lo) {
                any = true;
                if (!visible(lo, p, Tk, P.causal, P.window) || !visible(hi - 1, p, Tk, P.causal, P.window) ||
                    (lo > 0 && visible(lo - 1, p, Tk, P.causal, P.window)) || visible(hi, p, Tk, P.causal, P.window)) {
                    if (bad++ < 5) std::printf("ends wrong at p=%lld Tk=%lld w=%d\n", (long long)p, (long long)Tk, P.window);
                }
                if (lo < first_lo) {
                    if (bad++ < 5) std::printf("a row sees a key before the first row's\n");
                }
                union_hi = hi > union_hi ? hi : union_hi;
            } else if (visible(lo, p, Tk, P.causal, P.window) || (lo > 0 && visible(lo - 1, p, Tk, P.causal, P.window))) {
                if (bad++ < 5) std::printf("empty interval but a visible key at p=%lld\n", (long long)p);
            }
        }
        // the last row's hi is the largest: the walk [first lo, last hi) covers every row's keys
        if (any && phi < union_hi) {
            if (bad++ < 5) std::printf("the last row's hi is not the largest\n");
        }
    }
    // The boundary tiles' bit form of a thread's interval [elo, ehi) of its
    // 64 keys: every interval, every key.
    for (int elo = 0; elo <= 64; ++elo)
        for (int ehi = 0; ehi <= 64; ++ehi) {
            const fa::KeyBits kb = fa::key_bits(elo, ehi);
            for (int e = 0; e < 64; ++e) {
                ++checked;
                if (kb.has(e) != (e >= elo && e < ehi)) {
                    if (bad++ < 5) std::printf("key bit %d of [%d, %d)\n", e, elo, ehi);
                }
            }
        }
    std::printf("checked %ld, failures %ld\n", checked, bad);
    return bad == 0 ? 0 : 1;
}
"""


def test_visible_range_matches_the_rule(tmp_path):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("no host C++ compiler")
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    inc = Path(nvcc).resolve().parent.parent / "include"
    if not (inc / "cuda_runtime.h").exists():
        pytest.skip("CUDA headers not found")
    src = tmp_path / "vis.cpp"
    src.write_text(_DRIVER)
    exe = tmp_path / "vis"
    subprocess.run([gxx, "-std=c++17", "-O2", "-fsanitize=undefined", "-fno-sanitize-recover=all", f"-I{_CSRC}",
                    f"-I{inc}", str(src), "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and "runtime error" not in r.stderr, r.stdout + r.stderr
    assert "failures 0" in r.stdout
