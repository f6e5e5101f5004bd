// Exact unsigned 64-bit division by a run-time invariant divisor, by multiplication.
//
// Method: T. Granlund and P. L. Montgomery, "Division by Invariant Integers using
// Multiplication", PLDI 1994, Figure 4.1 (unsigned division, N = 64 bits):
//   l   = ceil(log2 d)
//   m'  = floor(2^N (2^l - d) / d) + 1
//   sh1 = min(l, 1), sh2 = max(l - 1, 0)
//   q   = SRL(t1 + SRL(n - t1, sh1), sh2),  t1 = MULUH(m', n)
// which equals floor(n / d) for every 0 <= n < 2^N and 1 <= d < 2^N.  The
// multiplier is computed once per divisor (by a 128-by-64-bit long division
// written here as plain shift-and-subtract); each division then costs one
// high multiply, an add, a subtract and two shifts.
//
// The header compiles both as CUDA and as plain C++ (for the host-side check).
#pragma once

#include <cstdint>

#ifndef __CUDACC__
#ifndef __host__
#define __host__
#endif
#ifndef __device__
#define __device__
#endif
#endif

namespace nest {

struct Divisor {
    uint64_t mul;
    uint32_t sh1, sh2;
};

__host__ __device__ inline uint64_t mulhi64(uint64_t a, uint64_t b) {
#ifdef __CUDA_ARCH__
    return __umul64hi(a, b);
#else
    return uint64_t((unsigned __int128)a * b >> 64);
#endif
}

// floor((hi * 2^64 + 0) / d) for hi < d.  Divisors below 2^41 take three long-division
// steps of 22, 21 and 21 quotient bits (the remainder stays below d, so the shifted
// remainder fits 64 bits): each step estimates its quotient digit with a float
// reciprocal (within a few units of the digit, which is below 2^22) and corrects it
// exactly with integer arithmetic.  Larger divisors go bit by bit.
__host__ __device__ inline uint64_t div128_by_64(uint64_t hi, uint64_t d) {
    if (d == 0) return 0;   // no divisor: never used (callers validate d >= 1 first)
    if (d < (uint64_t(1) << 41)) {
        const float rd = 1.0f / float(d);
        uint64_t q = 0, r = hi;
        const int step[3] = {22, 21, 21};
        for (int k = 0; k < 3; k++) {
            r <<= step[k];                                       // r < 2^63
            float est = float(r) * rd;
            est = est < 0.0f ? 0.0f : est;
            uint64_t qk = uint64_t(est);                         // < 2^22 + a few
            int64_t rem = int64_t(r - qk * d);   // the true difference is a few d: wraps exactly
            while (rem < 0) {
                qk--;
                rem += int64_t(d);
            }
            while (rem >= int64_t(d)) {
                qk++;
                rem -= int64_t(d);
            }
            r = uint64_t(rem);
            q = (q << step[k]) | qk;
        }
        return q;
    }
    uint64_t q = 0, r = hi;  // invariant r < d
    for (int bit = 63; bit >= 0; --bit) {
        const bool carry = (r >> 63) != 0;  // r * 2 overflows 64 bits
        r <<= 1;                             // next dividend bit is 0
        if (carry || r >= d) {
            r -= d;
            q |= uint64_t(1) << bit;
        }
    }
    return q;
}

__host__ __device__ inline Divisor make_divisor(uint64_t d) {
    Divisor v;
    // l = ceil(log2 d)
#ifdef __CUDA_ARCH__
    const uint32_t l = d <= 1 ? 0u : uint32_t(64 - __clzll((long long)(d - 1)));
#else
    const uint32_t l = d <= 1 ? 0u : uint32_t(64 - __builtin_clzll(d - 1));
#endif
    // m' = floor(2^64 (2^l - d) / d) + 1; (2^l - d) < d so the quotient fits 64 bits
    const uint64_t top = l == 64 ? uint64_t(0) - d : (uint64_t(1) << l) - d;
    v.mul = div128_by_64(top, d) + 1;
    v.sh1 = l < 1 ? l : 1;
    v.sh2 = l > 1 ? l - 1 : 0;
    return v;
}

__host__ __device__ inline uint64_t divide(uint64_t n, const Divisor &v) {
    const uint64_t t1 = mulhi64(v.mul, n);
    return (t1 + ((n - t1) >> v.sh1)) >> v.sh2;
}

// ceil(n / d) for n + d - 1 < 2^64.
__host__ __device__ inline uint64_t divide_up(uint64_t n, uint64_t d, const Divisor &v) {
    return divide(n + d - 1, v);
}

}  // namespace nest
