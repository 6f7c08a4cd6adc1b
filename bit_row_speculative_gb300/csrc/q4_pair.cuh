// Float pairs: an unevaluated sum hi + lo of two floats carrying about 48
// significant bits, with error-free transformations (two-sum, fma-split
// products) on the single-precision pipes; and the exponential to that
// precision.  Used where a result must round like a double-precision one
// without GB300's narrow FP64 units: the glue's near-tie outputs and the
// sampling epilogue's probabilities.
#pragma once

#include <cstdint>

namespace q4 {
namespace pair {

struct fpair {
    float hi, lo;
};

__device__ __forceinline__ fpair fast_two_sum(float a, float b) {   // |a| >= |b|
    const float s = __fadd_rn(a, b);
    return {s, __fsub_rn(b, __fsub_rn(s, a))};
}

__device__ __forceinline__ fpair two_sum(float a, float b) {
    const float s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    return {s, __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb))};
}

__device__ __forceinline__ fpair pair_add(fpair a, fpair b) {
    fpair s = two_sum(a.hi, b.hi);
    return fast_two_sum(s.hi, __fadd_rn(s.lo, __fadd_rn(a.lo, b.lo)));
}

__device__ __forceinline__ fpair pair_mul(fpair a, fpair b) {
    const float p = __fmul_rn(a.hi, b.hi);
    const float e = __fadd_rn(__fmaf_rn(a.hi, b.hi, -p), __fadd_rn(__fmul_rn(a.hi, b.lo), __fmul_rn(a.lo, b.hi)));
    return fast_two_sum(p, e);
}

__device__ __forceinline__ fpair pair_mul_f(fpair a, float b) {
    const float p = __fmul_rn(a.hi, b);
    return fast_two_sum(p, __fadd_rn(__fmaf_rn(a.hi, b, -p), __fmul_rn(a.lo, b)));
}

__device__ __forceinline__ fpair f_div_pair(float a, fpair d) {   // a / d
    const float q1 = __fdiv_rn(a, d.hi);
    const float r = __fsub_rn(__fmaf_rn(-q1, d.hi, a), __fmul_rn(q1, d.lo));
    return fast_two_sum(q1, __fdiv_rn(r, d.hi));
}

__device__ __forceinline__ fpair pair_div_f(fpair a, float b) {  // a / b
    const float q1 = __fdiv_rn(a.hi, b);
    const float r = __fadd_rn(__fmaf_rn(-q1, b, a.hi), a.lo);
    return fast_two_sum(q1, __fdiv_rn(r, b));
}

__device__ __forceinline__ fpair pair_div(fpair a, fpair b) {     // a / b
    const float q1 = __fdiv_rn(a.hi, b.hi);
    const float r = __fsub_rn(__fadd_rn(__fmaf_rn(-q1, b.hi, a.hi), a.lo), __fmul_rn(q1, b.lo));
    return fast_two_sum(q1, __fdiv_rn(r, b.hi));
}

// exp(x) as a float pair, relative error about 1e-14 for -60 <= x <= 88 (below
// -60 the low part turns subnormal; exp(x) < 1e-26 there).  x = k ln2 + r with
// ln 2 split into three floats (k * L1 exact), exp(r) by its Taylor series:
// the terms of order 7 and up in float, the rest in pairs.
__device__ __forceinline__ fpair exp_pair(float x) {
    const float kL1 = 0.693145751953125f;           // 16 significant bits
    const float kL2 = __uint_as_float(0x35bfbe8eu);  // ln 2 - L1, rounded
    const float kL3 = __uint_as_float(0x29778000u);  // ln 2 - L1 - L2, rounded
    const float k = rintf(__fmul_rn(x, 1.44269504f));
    const float t = __fsub_rn(x, __fmul_rn(k, kL1));  // exact
    const float p = __fmul_rn(k, kL2);
    const float pe = __fmaf_rn(k, kL2, -p);
    fpair r = two_sum(t, -p);
    r = fast_two_sum(r.hi, __fsub_rn(__fsub_rn(r.lo, pe), __fmul_rn(k, kL3)));
    // 1/n!: n = 7..13 as floats, n = 0..6 as pairs
    const float c_hi[7] = {__uint_as_float(0x2f309231u), __uint_as_float(0x310f76c7u), __uint_as_float(0x32d7322bu),
                            __uint_as_float(0x3493f27eu), __uint_as_float(0x3638ef1du), __uint_as_float(0x37d00d01u),
                            __uint_as_float(0x39500d01u)};
    float sf = c_hi[0];
#pragma unroll
    for (int n = 1; n < 7; ++n) sf = __fmaf_rn(sf, r.hi, c_hi[n]);   // orders 13 .. 7
    const uint32_t ph[7] = {0x3ab60b61u, 0x3c088889u, 0x3d2aaaabu, 0x3e2aaaabu, 0x3f000000u, 0x3f800000u, 0x3f800000u};
    const uint32_t pl[7] = {0xae13e93fu, 0xafeeeeefu, 0xb0aaaaabu, 0xb1aaaaabu, 0u, 0u, 0u};
    fpair S = {sf, 0.0f};
#pragma unroll
    for (int n = 0; n < 7; ++n)                                       // orders 6 .. 0
        S = pair_add(pair_mul(S, r), fpair{__uint_as_float(ph[n]), __uint_as_float(pl[n])});
    const float sc = __int_as_float(((int)k + 127) << 23);           // 2^k (-87 <= k <= 127 here)
    return {__fmul_rn(S.hi, sc), __fmul_rn(S.lo, sc)};
}

}  // namespace pair
}  // namespace q4
