// dfloat.cuh -- double-float arithmetic on the FP32 pipes: a value is an
// unevaluated sum hi + lo of two floats (~48 significant bits).  GB300's fp64
// pipe is narrow, so the running sums, scans and normalisers of the accept
// kernels use these instead of fp64.  The building blocks are the error-free
// transformations of Knuth (two-sum) and Dekker (fast two-sum) and the
// FMA-based exact product; df_exp_diff is a Cody-Waite reduction with a
// Taylor polynomial, described at the function.
#pragma once
#include <cuda_runtime.h>

namespace magicdec {

struct dflt {
    float hi, lo;
};

__device__ __forceinline__ dflt quick_two_sum(float a, float b) {
    const float s = a + b;
    return {s, b - (s - a)};
}

__device__ __forceinline__ dflt two_sum(float a, float b) {
    const float s = a + b;
    const float bb = s - a;
    return {s, (a - (s - bb)) + (b - bb)};
}

__device__ __forceinline__ dflt df_add_f(dflt a, float b) {
    dflt s = two_sum(a.hi, b);
    s.lo += a.lo;
    return quick_two_sum(s.hi, s.lo);
}

__device__ __forceinline__ dflt df_add(dflt a, dflt b) {
    dflt s = two_sum(a.hi, b.hi);
    s.lo += a.lo + b.lo;
    return quick_two_sum(s.hi, s.lo);
}

// float x double-float -> double-float
__device__ __forceinline__ dflt df_mul_f(float a, dflt b) {
    const float p = a * b.hi;
    const float e = fmaf(a, b.hi, -p) + a * b.lo;
    return quick_two_sum(p, e);
}

__device__ __forceinline__ dflt df_from_double(double x) {
    const float hi = (float)x;
    return {hi, (float)(x - (double)hi)};
}

__device__ __forceinline__ double df_to_double(dflt a) { return (double)a.hi + (double)a.lo; }

// Warp sum of double-float values in a fixed butterfly order (fp32 pipe only).
__device__ __forceinline__ dflt warp_sum_df(dflt a) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        dflt b;
        b.hi = __shfl_xor_sync(0xffffffffu, a.hi, o);
        b.lo = __shfl_xor_sync(0xffffffffu, a.lo, o);
        a = df_add(a, b);
    }
    return a;
}

__device__ __forceinline__ dflt df_sub(dflt a, dflt b) { return df_add(a, dflt{-b.hi, -b.lo}); }

__device__ __forceinline__ dflt df_mul(dflt a, dflt b) {
    const float p = a.hi * b.hi;
    return quick_two_sum(p, fmaf(a.hi, b.hi, -p) + (a.hi * b.lo + a.lo * b.hi));
}

// a / b by long division in double-float (as in Bailey's double-double
// library): a single-precision quotient digit, the exact remainder, and two
// correction digits from it; ~1e-14 relative.
__device__ __forceinline__ dflt df_div(dflt a, dflt b) {
    const float q1 = a.hi / b.hi;
    const dflt r1 = df_sub(a, df_mul_f(q1, b));
    const float q2 = r1.hi / b.hi;
    const dflt r2 = df_sub(r1, df_mul_f(q2, b));
    const float q3 = r2.hi / b.hi;
    return df_add_f(quick_two_sum(q1, q2), q3);
}

// exp(a - b) for fp32 a <= b as a double-float on the FP32 pipes: within
// 1e-11 relative down to exp(-70); below that the low part is subnormal and
// the error stays under an absolute 2e-38.  The difference as an exact
// double-float pair; Cody-Waite
// reduction r = (a - b) - k ln 2 with ln 2 split into a 15-bit head (so k
// times it is exact) and a single-precision tail; exp(r), |r| <= ln2 / 2, by
// its Taylor series to degree 11 (remainder below 1e-14) evaluated by Horner's
// rule in double-float, the coefficients 1/n! as double-float pairs; then the
// exact scaling by 2^k.  Differences below -87 (exp below 1e-38) give 0.
__device__ __forceinline__ dflt df_exp_diff(float a, float b) {
    const dflt d = two_sum(a, -b);
    if (d.hi < -87.f) return dflt{0.f, 0.f};
    constexpr float kLn2Hi = 0x1.62e4p-1f, kLn2Lo = 0x1.7f7d1cp-20f;
    const float k = rintf(d.hi * 1.4426950408889634f);   // log2(e)
    const float tl = k * kLn2Lo, tle = fmaf(k, kLn2Lo, -tl);         // k * tail, exactly
    dflt r = two_sum(d.hi, -k * kLn2Hi);                              // exact
    r = df_add(r, dflt{-tl, -tle});
    r = df_add_f(r, d.lo);
    constexpr float C[12][2] = {{1.f, 0.f}, {1.f, 0.f}, {0.5f, 0.f},
                                {0x1.555556p-3f, -0x1.555556p-28f}, {0x1.555556p-5f, -0x1.555556p-30f},
                                {0x1.111112p-7f, -0x1.dddddep-32f}, {0x1.6c16c2p-10f, -0x1.27d27ep-35f},
                                {0x1.a01a02p-13f, -0x1.7f97fap-39f}, {0x1.a01a02p-16f, -0x1.7f97fap-42f},
                                {0x1.71de3ap-19f, 0x1.55b1ccp-45f}, {0x1.27e4fcp-22f, -0x1.10ec14p-47f},
                                {0x1.ae6456p-26f, 0x1.fd5138p-52f}};
    dflt e = {C[11][0], C[11][1]};
#pragma unroll
    for (int n = 10; n >= 0; --n) e = df_add(df_mul(e, r), dflt{C[n][0], C[n][1]});
    const float scale = __int_as_float((127 + (int)k) << 23);         // 2^k, k in [-126, 0]
    return {e.hi * scale, e.lo * scale};
}

// Order of normalised double-float values (|lo| at most half an ulp of hi).
__device__ __forceinline__ bool df_lt(dflt a, dflt b) { return a.hi < b.hi || (a.hi == b.hi && a.lo < b.lo); }
__device__ __forceinline__ bool df_le(dflt a, dflt b) { return a.hi < b.hi || (a.hi == b.hi && a.lo <= b.lo); }
__device__ __forceinline__ bool df_positive(dflt a) { return a.hi > 0.f || (a.hi == 0.f && a.lo > 0.f); }

__device__ __forceinline__ dflt df_shfl_up(dflt a, int o) {
    return {__shfl_up_sync(0xffffffffu, a.hi, o), __shfl_up_sync(0xffffffffu, a.lo, o)};
}
__device__ __forceinline__ dflt df_shfl(dflt a, int src) {
    return {__shfl_sync(0xffffffffu, a.hi, src), __shfl_sync(0xffffffffu, a.lo, src)};
}

}  // namespace magicdec
