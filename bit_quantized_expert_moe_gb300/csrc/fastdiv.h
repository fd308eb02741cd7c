// Division of unsigned 32-bit values n < 2^31 by a divisor fixed per launch,
// as one multiply-high, an add and a shift: T. Granlund and P. L. Montgomery,
// "Division by Invariant Integers using Multiplication" (PLDI 1994), the
// unsigned case with l = ceil(log2 d):
//     m = floor(2^32 (2^l - d) / d) + 1,    floor(n / d) = (mulhi(m, n) + n) >> l.
// (mulhi(m, n) <= n, so the sum stays below 2^32 for n < 2^31.)  The constants
// are computed on the host; the quotient is taken on either side.
#pragma once

#include <cstdint>

#ifdef __CUDACC__
#define MOE_HD __host__ __device__ __forceinline__
#else
#define MOE_HD inline
#endif

namespace moe {

struct FastDiv {
    uint32_t d, m, l;
};

inline FastDiv make_fastdiv(uint32_t d) {
    FastDiv f{d, 0u, 0u};
    if (d == 0) return f;
    uint32_t l = 0;
    while (l < 32 && (1ull << l) < d) ++l;
    f.l = l;
    f.m = (uint32_t)((((1ull << l) - d) << 32) / d + 1);
    return f;
}

MOE_HD uint32_t fd_div(uint32_t n, FastDiv f) {
#ifdef __CUDA_ARCH__
    const uint32_t hi = __umulhi(n, f.m);
#else
    const uint32_t hi = (uint32_t)(((uint64_t)n * f.m) >> 32);
#endif
    return (hi + n) >> f.l;
}

// quotient and remainder
MOE_HD uint32_t fd_divmod(uint32_t n, FastDiv f, uint32_t* r) {
    const uint32_t q = fd_div(n, f);
    *r = n - q * f.d;
    return q;
}

}  // namespace moe
