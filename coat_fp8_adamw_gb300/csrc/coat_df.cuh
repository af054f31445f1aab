// coat_df.cuh -- double-float ("hi + lo" pair of fp32) arithmetic for the few
// per-group quantities whose fp32 rounding would be visible: the exponent k
// (rounded to fp32 once, from a ~2^-44-accurate value), the scale S, the
// dequantization factor P, and exact re-evaluation of a group's extreme
// moments.
//
// Everything here is built from IEEE-exact operations only -- add, multiply,
// fused multiply-add and divide with round-to-nearest-even -- so the same
// code gives bit-identical results on the device and on the host (where the
// CPU tests exercise it).  The error-free transformations are Knuth's
// TwoSum, Dekker's FastTwoSum and the FMA-based TwoProduct; log2 uses a
// 64-entry table of log2(c_j) with the atanh series of ln(u/c_j); exp2 uses a
// 32-entry table of 2^(j/32) with the Taylor series of e^a on |a| < 0.011.
// The tables are generated in float64 by gen_tables.py.
#pragma once

#include <cstdint>
#include <cstring>

#if defined(__CUDACC__)
#include <cuda_runtime.h>
#define COAT_HD __host__ __device__ __forceinline__
#else
#include <cmath>
#define COAT_HD inline
#endif

namespace coat {
namespace df {

struct F2 {
    float hi, lo;
};

// --- IEEE primitives that the device compiler must not contract or reorder ---
COAT_HD float add(float a, float b) {
#if defined(__CUDA_ARCH__)
    return __fadd_rn(a, b);
#else
    return a + b;
#endif
}
COAT_HD float sub(float a, float b) {
#if defined(__CUDA_ARCH__)
    return __fsub_rn(a, b);
#else
    return a - b;
#endif
}
COAT_HD float mul(float a, float b) {
#if defined(__CUDA_ARCH__)
    return __fmul_rn(a, b);
#else
    return a * b;
#endif
}
COAT_HD float fma(float a, float b, float c) {
#if defined(__CUDA_ARCH__)
    return __fmaf_rn(a, b, c);
#else
    return std::fma(a, b, c);
#endif
}
COAT_HD float div(float a, float b) {
#if defined(__CUDA_ARCH__)
    return __fdiv_rn(a, b);
#else
    return a / b;
#endif
}
COAT_HD float rint(float x) {
#if defined(__CUDA_ARCH__)
    return rintf(x);
#else
    return std::nearbyint(x);
#endif
}
COAT_HD uint32_t bits(float x) {
#if defined(__CUDA_ARCH__)
    return __float_as_uint(x);
#else
    uint32_t u;
    std::memcpy(&u, &x, 4);
    return u;
#endif
}
COAT_HD float from_bits(uint32_t u) {
#if defined(__CUDA_ARCH__)
    return __uint_as_float(u);
#else
    float x;
    std::memcpy(&x, &u, 4);
    return x;
#endif
}

// x * 2^n for integer n, exact whenever the result is a normal float
// (two power-of-two factors so that n in [-252, 254] is covered; beyond that
// range the result saturates to 0 or infinity for |x| in [0.5, 2)).
COAT_HD float scale2(float x, int n) {
    n = n < -252 ? -252 : (n > 254 ? 254 : n);
    const int n1 = n / 2, n2 = n - n / 2;
    return mul(mul(x, from_bits((uint32_t)(n1 + 127) << 23)), from_bits((uint32_t)(n2 + 127) << 23));
}

// --- error-free transformations ---
COAT_HD F2 two_sum(float a, float b) {
    const float s = add(a, b);
    const float bb = sub(s, a);
    const float e = add(sub(a, sub(s, bb)), sub(b, bb));
    return {s, e};
}
COAT_HD F2 fast_two_sum(float a, float b) {  // requires exponent(a) >= exponent(b)
    const float s = add(a, b);
    return {s, sub(b, sub(s, a))};
}
COAT_HD F2 two_prod(float a, float b) {
    const float p = mul(a, b);
    return {p, fma(a, b, -p)};
}

// (a + b) for double-floats, normalized
COAT_HD F2 add2(F2 a, F2 b) {
    const F2 s = two_sum(a.hi, b.hi);
    return fast_two_sum(s.hi, add(s.lo, add(a.lo, b.lo)));
}
COAT_HD F2 neg2(F2 a) { return {-a.hi, -a.lo}; }

// a * b for a double-float and a float
COAT_HD F2 mul21(F2 a, float b) {
    const F2 p = two_prod(a.hi, b);
    return fast_two_sum(p.hi, fma(a.lo, b, p.lo));
}
// a * b for two double-floats
COAT_HD F2 mul22(F2 a, F2 b) {
    const F2 p = two_prod(a.hi, b.hi);
    return fast_two_sum(p.hi, fma(a.hi, b.lo, fma(a.lo, b.hi, p.lo)));
}
// a / b for a double-float and a float
COAT_HD F2 div21(F2 a, float b) {
    const float q = div(a.hi, b);
    const float r = add(fma(-q, b, a.hi), a.lo);  // a.hi - q b is exact for a rounded quotient
    return fast_two_sum(q, div(r, b));
}
// a / b for two double-floats as an unrounded pair q + c (|c| <= ulp(q))
COAT_HD F2 div22_parts(F2 a, F2 b) {
    const float q = div(a.hi, b.hi);
    const float r = sub(add(fma(-q, b.hi, a.hi), a.lo), mul(q, b.lo));
    return {q, div(r, b.hi)};
}
// a / b for two double-floats, rounded once to the nearest float
COAT_HD float div22_rn(F2 a, F2 b) {
    const F2 p = div22_parts(a, b);
    return add(p.hi, p.lo);
}

// --- constants (double-float) ---
struct Tables {
    const float* log2c_hi;  // [64] log2(1 + (2j+1)/128)
    const float* log2c_lo;
    const float* exp2j_hi;  // [33] 2^(j/32), j = -16..16 (index j + 16)
    const float* exp2j_lo;
};
constexpr float kInvLn2Hi = 1.44269502162933349609375f;      // 1/ln 2 = hi + lo
constexpr float kInvLn2Lo = 1.925963033500011079013347625732421875e-08f;
constexpr float kLn2Hi = 0.693147182464599609375f;           // ln 2 = hi + lo
constexpr float kLn2Lo = -1.9046542121259336e-09f;

// log2(x) for finite x > 0 (normal or subnormal), |error| <~ 2^-46 + 2^-47 |log2 x|.
COAT_HD F2 log2_df(float x, const Tables& t) {
    uint32_t b = bits(x);
    int ex = (int)((b >> 23) & 0xFFu);
    if (ex == 0) {  // subnormal: scale by 2^24 (exact)
        b = bits(mul(x, 16777216.0f));
        ex = (int)((b >> 23) & 0xFFu) - 24;
    }
    const int e = ex - 127;
    const uint32_t j = (b >> 17) & 63u;
    const float u = from_bits((b & 0x007FFFFFu) | 0x3F800000u);
    const float c = from_bits(0x3F800000u | (j << 17) | (1u << 16));  // 1 + (2j+1)/128
    // s = (u - c) / (u + c), |s| <= 2^-8
    const float num = sub(u, c);                 // exact (Sterbenz)
    const F2 den = fast_two_sum(u, c);           // same binade: exact split
    const float s = div(num, den.hi);
    const float r = fma(-s, den.lo, fma(-s, den.hi, num));
    const float s_lo = div(r, den.hi);
    // ln(u/c) = 2 atanh(s) = 2s + (2/3)s^3 + (2/5)s^5 + O(s^7)
    const float s2 = mul(s, s);
    const float poly = mul(mul(s, s2), fma(0.4f, s2, 0.666666686534881591796875f));
    const F2 ln_uc = fast_two_sum(mul(2.0f, s), add(mul(2.0f, s_lo), poly));
    // to base 2
    const F2 l2 = mul22(ln_uc, F2{kInvLn2Hi, kInvLn2Lo});
    // + log2(c_j) + e
    const F2 lc = {t.log2c_hi[j], t.log2c_lo[j]};
    const F2 frac = add2(lc, l2);                  // in [0, 1)
    const F2 whole = two_sum((float)e, frac.hi);
    return two_sum(whole.hi, add(whole.lo, frac.lo));
}

// 2^z for a double-float z as 2^n (m.hi + m.lo), with m.hi + m.lo in about
// [0.7, 1.42] not yet rounded: the caller rounds m once and scales it by 2^n.
COAT_HD F2 exp2_df_parts(F2 z, const Tables& t, int& n_out) {
    const float n = rint(z.hi);
    const F2 f = two_sum(sub(z.hi, n), z.lo);      // |f| <= 0.5 + tiny
    const float jf = rint(mul(f.hi, 32.0f));       // -16..16 for a normalized z
    // clamped so that no input (even a non-normalized or non-finite one) can
    // index outside the 33-entry table
    const int j0 = (int)jf;
    const int j = j0 < -16 ? -16 : (j0 > 16 ? 16 : j0);
    const F2 r = fast_two_sum(sub(f.hi, mul(jf, 0.03125f)), f.lo);  // |r| <= 1/64
    // a = r ln 2
    const F2 a = mul22(r, F2{kLn2Hi, kLn2Lo});
    // e^a - 1 = a + a^2/2 + a^3/6 + a^4/24 + a^5/120 (|a| < 0.011: next term < 2^-48)
    const F2 sq = two_prod(a.hi, a.hi);
    const F2 s1 = fast_two_sum(a.hi, mul(sq.hi, 0.5f));
    const float cube = mul(mul(a.hi, sq.hi),
                           fma(a.hi, fma(a.hi, 0.008333333767950534820556640625f,
                                         0.0416666679084300994873046875f),
                               0.16666667163372039794921875f));
    const float rest = add(add(add(s1.lo, a.lo), fma(0.5f, sq.lo, mul(a.hi, a.lo))), cube);
    const F2 em1 = fast_two_sum(s1.hi, rest);
    // 2^f = T_j (1 + em1)
    const F2 T = {t.exp2j_hi[j + 16], t.exp2j_lo[j + 16]};
    const F2 p = two_prod(T.hi, em1.hi);
    const F2 h = two_sum(T.hi, p.hi);
    const float lo = add(add(h.lo, p.lo), fma(T.hi, em1.lo, fma(T.lo, em1.hi, T.lo)));
    n_out = (int)n;
    return {h.hi, lo};
}

// 2^z for a double-float z, rounded once to float (normal results).
COAT_HD float exp2_df(F2 z, const Tables& t) {
    int n = 0;
    const F2 m = exp2_df_parts(z, t, n);
    return scale2(add(m.hi, m.lo), n);              // rounded once
}

// round-to-nearest of a*b + c*d for floats, via error-free products and sum
COAT_HD float dot2_rn(float a, float b, float c, float d) {
    const F2 p = two_prod(a, b);
    const F2 q = two_prod(c, d);
    const F2 s = two_sum(p.hi, q.hi);
    return add(s.hi, add(s.lo, add(p.lo, q.lo)));
}

}  // namespace df
}  // namespace coat
