// fastdiv.h -- integer division by a divisor that is fixed for a launch, as
// one widening multiply and one shift (Granlund and Montgomery, "Division by
// invariant integers using multiplication", PLDI 1994, the round-up
// multiplier).
//
// For a divisor 1 <= d < 2^31, let s be the least integer with d <= 2^s,
// p = 31 + s and m = ceil(2^p / d).  Then 2^31 <= m < 2^32 and
//     floor(n / d) == (n * m) >> p   for every 0 <= n < 2^31:
// n m / 2^p = n / d + n e / (d 2^p) with e = m d - 2^p in [0, d), and
// n e < 2^31 2^s = 2^p, so the added fraction stays below 1 / d and cannot
// carry floor(n / d) to the next integer.
//
// Plain C++ (no CUDA types) so that the host, the device code and a CPU test
// program share this one definition.
#pragma once

#if defined(__CUDACC_RTC__)
// the runtime compiler has no host headers; rtc_compat.cuh supplies the types
#else
#include <cstdint>
#endif

#if defined(__CUDACC__) || defined(__CUDACC_RTC__)
#define FL_FASTDIV_FN __host__ __device__ __forceinline__
#else
#define FL_FASTDIV_FN inline
#endif

namespace fl {

struct FastDiv {
    int32_t d;  // the divisor
    uint32_t m; // ceil(2^p / d)
    uint32_t p; // 31 + ceil(log2 d)
};

// d must lie in [1, 2^31); callers check it.
FL_FASTDIV_FN FastDiv make_fastdiv(int32_t d)
{
    uint32_t s = 0;
    while ((uint64_t(1) << s) < uint64_t(d))
        ++s;
    FastDiv f;
    f.d = d;
    f.p = 31 + s;
    f.m = uint32_t(((uint64_t(1) << f.p) + uint64_t(d) - 1) / uint64_t(d));
    return f;
}

// floor(n / f.d) for 0 <= n < 2^31.
FL_FASTDIV_FN int32_t fast_div(int32_t n, const FastDiv &f)
{
    return int32_t((uint64_t(uint32_t(n)) * f.m) >> f.p);
}

} // namespace fl
