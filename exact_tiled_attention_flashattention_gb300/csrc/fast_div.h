// fast_div.h -- quotient and remainder of 32-bit indices by a divisor fixed
// at launch, as one multiply-high, one add and one shift.
//
// Method: Granlund and Montgomery, "Division by invariant integers using
// multiplication" (PLDI 1994), the unsigned case.  With s = ceil(log2 d) and
// M = floor(2^(32+s) / d) + 1, which lies in (2^32, 2^33], floor(n / d) =
// floor(n * M / 2^(32+s)) for every 32-bit n, because M d - 2^(32+s) <= d <=
// 2^s.  M does not fit in 32 bits; storing m = M - 2^32 gives
// floor(n / d) = (umulhi(n, m) + n) >> s, whose sum does not overflow for
// n < 2^31 (umulhi(n, m) < n).  The kernels' unit and row indices stay below
// 2^31 (the host rejects larger grids).
#pragma once

#include <cstdint>

#ifdef __CUDACC__
#define FA_HOST_DEVICE __host__ __device__
#else
#define FA_HOST_DEVICE
#endif

namespace fa {

struct FastDiv {
    uint32_t d, m, s;

    // d >= 1 and d < 2^31.
    static FA_HOST_DEVICE FastDiv make(uint32_t d) {
        FastDiv f{};
        f.d = d;
        f.s = 0;
        while ((uint64_t(1) << f.s) < d) ++f.s;
        f.m = (uint32_t)(((uint64_t(1) << 32) * ((uint64_t(1) << f.s) - d)) / d + 1);
        return f;
    }

    // n < 2^31.
    FA_HOST_DEVICE uint32_t div(uint32_t n) const {
#ifdef __CUDA_ARCH__
        const uint32_t hi = __umulhi(n, m);
#else
        const uint32_t hi = (uint32_t)(((uint64_t)n * m) >> 32);
#endif
        return (hi + n) >> s;
    }

    FA_HOST_DEVICE uint32_t mod(uint32_t n) const { return n - div(n) * d; }
};

}  // namespace fa
