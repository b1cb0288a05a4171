"""Host check of the kernels' division by launch constants (csrc/fast_div.h).

The header is compiled on the host with g++ and compared with the machine's
own division: every divisor up to 4096 against dividends near 0, near
multiples of the divisor and near 2^31, every divisor up to 2^16 on random
dividends, and divisors near powers of two up to 2^30.  The kernels take the
same code path (only the multiply-high instruction differs in name).
"""
import os
import shutil
import subprocess

import pytest

_ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
_HDR = os.path.join(_ROOT, "exact_tiled_attention_flashattention_gb300", "csrc")

_SRC = r"""
#include <cstdint>
#include <cstdio>
#include "fast_div.h"
static uint64_t state = 0x9e3779b97f4a7c15ull;
static uint32_t next() {  // xorshift64*
    state ^= state >> 12; state ^= state << 25; state ^= state >> 27;
    return (uint32_t)((state * 0x2545f4914f6cdd1dull) >> 33);  // 31 bits
}
static long bad = 0, checked = 0;
static void check(const fa::FastDiv &f, uint32_t n) {
    ++checked;
    if (f.div(n) != n / f.d || f.mod(n) != n % f.d) {
        if (bad < 5) std::printf("FAIL d=%u n=%u: %u %u\n", f.d, n, f.div(n), f.mod(n));
        ++bad;
    }
}
int main() {
    const uint32_t top = 0x7fffffffu;
    for (uint32_t d = 1; d <= 4096; ++d) {
        const fa::FastDiv f = fa::FastDiv::make(d);
        for (uint32_t n = 0; n < 3 * d + 5; ++n) check(f, n);
        for (uint32_t k = 0; k < 64; ++k) check(f, top - k);
        for (uint32_t k = 1; k < 200; ++k) {
            const uint64_t q = (uint64_t)next() % (top / d + 1);
            const uint64_t base = q * d;
            for (int64_t e = -1; e <= 1; ++e) {
                const int64_t n = (int64_t)base + e;
                if (n >= 0 && n <= top) check(f, (uint32_t)n);
            }
        }
    }
    for (uint32_t d = 4097; d <= 65536; ++d) {
        const fa::FastDiv f = fa::FastDiv::make(d);
        for (int k = 0; k < 40; ++k) check(f, next());
        check(f, top);
        check(f, d - 1);
        check(f, d);
    }
    for (int p = 2; p <= 30; ++p)
        for (int64_t e = -3; e <= 3; ++e) {
            const fa::FastDiv f = fa::FastDiv::make((uint32_t)((int64_t(1) << p) + e));
            for (int k = 0; k < 20000; ++k) check(f, next());
            check(f, top);
        }
    std::printf("checked %ld, failures %ld\n", checked, bad);
    return bad == 0 ? 0 : 1;
}
"""


def test_fast_div_matches_division(tmp_path):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("no host C++ compiler")
    src = tmp_path / "fd.cpp"
    src.write_text(_SRC)
    exe = tmp_path / "fd"
    subprocess.run([gxx, "-O2", "-std=c++17", f"-I{_HDR}", str(src), "-o", str(exe)], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "failures 0" in r.stdout
