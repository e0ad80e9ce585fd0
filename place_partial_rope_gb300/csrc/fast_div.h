// fast_div.h -- unsigned 32-bit division by a run-time invariant divisor
// with one multiply-high, one add and one shift.
//
// Method: T. Granlund and P. L. Montgomery, "Division by Invariant Integers
// using Multiplication" (PLDI 1994), section 4, unsigned division with an
// N+1-bit multiplier: for a divisor d in [1, 2^32), let l = ceil(log2 d) and
// m = floor(2^32 * (2^l - d) / d) + 1 (which fits 32 bits).  Then for every
// n in [0, 2^32): n / d = (mulhi(m, n) + n) >> l, where the sum is formed in
// 64 bits so it cannot overflow.
#pragma once
#include <stdint.h>

#if defined(__CUDACC__)
#define ROPE_HD __host__ __device__ __forceinline__
#else
#define ROPE_HD inline
#endif

namespace rope {

struct FastDiv {
    uint32_t d;  // divisor
    uint32_t m;  // magic multiplier
    uint32_t l;  // shift

    static FastDiv make(uint32_t divisor) {
        FastDiv f;
        f.d = divisor;
        uint32_t l = 0;
        while (l < 32 && (uint64_t(1) << l) < divisor) ++l;
        f.l = l;
        const uint64_t num = (uint64_t(1) << 32) * ((uint64_t(1) << l) - divisor);
        f.m = uint32_t(num / divisor + 1);
        return f;
    }

    ROPE_HD uint32_t div(uint32_t n) const {
#if defined(__CUDA_ARCH__)
        const uint32_t hi = __umulhi(m, n);
#else
        const uint32_t hi = uint32_t((uint64_t(m) * n) >> 32);
#endif
        return uint32_t((uint64_t(hi) + n) >> l);
    }

    // quotient and remainder
    ROPE_HD void divmod(uint32_t n, uint32_t& q, uint32_t& r) const {
        q = div(n);
        r = n - q * d;
    }
};

}  // namespace rope
