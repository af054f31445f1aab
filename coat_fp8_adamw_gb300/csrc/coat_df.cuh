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
// TwoSum, Dekker's FastTwoSum and the FMA-based TwoProduct; log2 reduces the
// significand u by a 9-bit reciprocal r_j of its interval (one of 256; then
// u r_j - 1 is exact in fp32, one FMA) and sums -log2 r_j (a 256-entry table)
// with the Taylor series of log2(1 + t) on |t| < 2^-8.45; exp2 uses a 32-entry table of
// 2^(j/32) with the Taylor series of e^a on |a| < 0.011.  The tables are
// generated in float64 by gen_tables.py.
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
    // one factor when 2^n is a normal float: the same single rounding
    if (n >= -126 && n <= 127) return mul(x, from_bits((uint32_t)(n + 127) << 23));
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
// 1 / b as a double-float with one division: q = RN(1/b), the exact remainder
// 1 - q b (one FMA), and its quotient by b formed as a product with q (a
// relative error of 2^-23 on a part below 2^-24 q).
COAT_HD F2 recip21(float b) {
    const float q = div(1.0f, b);
    const float r = fma(-q, b, 1.0f);
    return fast_two_sum(q, mul(r, q));
}
// a / b for two double-floats as an unrounded pair q + c, with 1 / a.hi given
// (a constant numerator): the correction r / b.hi is formed as r q (1 / a.hi),
// within a relative 2^-22 of it; |c| <= ulp(q).
COAT_HD F2 div22_parts_k(F2 a, float rcp_a_hi, F2 b) {
    const float q = div(a.hi, b.hi);
    const float r = sub(add(fma(-q, b.hi, a.hi), a.lo), mul(q, b.lo));
    return {q, mul(r, mul(q, rcp_a_hi))};
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
// One entry of the log2 reduction table: -log2 r_j (double-float).
struct alignas(8) LogEntry {
    float nl_hi, nl_lo;
};
struct Tables {
    const LogEntry* logr;   // [256], interval j of the significand (top 8 bits)
    const float* exp2j_hi;  // [33] 2^(j/32), j = -16..16 (index j + 16)
    const float* exp2j_lo;
};
constexpr float kInvLn2Hi = 1.44269502162933349609375f;      // 1/ln 2 = hi + lo
constexpr float kInvLn2Lo = 1.925963033500011079013347625732421875e-08f;
constexpr float kLn2Hi = 0.693147182464599609375f;           // ln 2 = hi + lo
constexpr float kLn2Lo = -1.9046542121259336e-09f;

// The Taylor coefficients of log2(1 + t) beyond the quadratic term, as floats:
// 1/(3 ln 2), -1/(4 ln 2), 1/(5 ln 2).
constexpr float kL2c3 = 0.480898350f;
constexpr float kL2c4 = -0.360673755f;
constexpr float kL2c5 = 0.288539022f;

// The reciprocal of the log2 reduction for interval j = 0..255 of the
// significand: r_j = rint(p(j)) / 512 with p a quartic close to
// 2^18 / (513 + 2j) (within 0.11), evaluated by FMAs, so r_j is a 9-bit value
// near 1 / (interval centre) with |u r_j - 1| < 2^-8.38 for every u in
// [1 + j/256, 1 + (j+1)/256); gen_tables.py reads the coefficients from here,
// repeats the evaluation exactly, checks that bound and tabulates -log2 r_j.
constexpr float kRecipP4 = 0x1.4a7454p-26f;
constexpr float kRecipP3 = -0x1.197b28p-16f;
constexpr float kRecipP2 = 0x1.bf7b12p-8f;
constexpr float kRecipP1 = -0x1.f7a158p+0f;
constexpr float kRecipP0 = 0x1.fee4eep+8f;
COAT_HD float log_recip(uint32_t j) {
    const float x = (float)j;
    const float p = fma(fma(fma(fma(kRecipP4, x, kRecipP3), x, kRecipP2), x, kRecipP1), x, kRecipP0);
    return mul(rint(p), 0.001953125f);
}

// log2(x) for finite x > 0 (normal or subnormal), |error| < 2^-46 + 2^-47 |log2 x|.
// x = 2^e u, u in [1, 2); with the table's r_j for the top 8 bits of u,
// t = u r_j - 1 is exact (|t| < 2^-8.38) and
//   log2 x = e - log2 r_j + c t - (c/2) t^2 + t^3 (c/3 - c t/4 + c t^2/5),
// c = 1/ln 2, truncated after t^5 (the next term is below 2^-52).  c t and
// (c/2) t^2 are carried as double-floats; the cubic tail (< 2^-26.2) in fp32.
COAT_HD F2 log2_df(float x, const Tables& t) {
    uint32_t b = bits(x);
    int ex = (int)((b >> 23) & 0xFFu);
    if (ex == 0) {  // subnormal: scale by 2^24 (exact)
        b = bits(mul(x, 16777216.0f));
        ex = (int)((b >> 23) & 0xFFu) - 24;
    }
    const uint32_t j = (b >> 15) & 255u;
    const LogEntry en = t.logr[j];
    const float u = from_bits((b & 0x007FFFFFu) | 0x3F800000u);
    const float w = fma(u, log_recip(j), -1.0f);          // t, exact
    const F2 a = two_prod(w, kInvLn2Hi);                  // c_hi t
    const F2 sq = two_prod(w, w);                         // t^2
    const F2 q = two_prod(sq.hi, mul(0.5f, kInvLn2Hi));   // (c_hi / 2) (t^2).hi
    const float tail = mul(mul(w, sq.hi), fma(fma(w, kL2c5, kL2c4), w, kL2c3));
    // the small parts: the low halves of the two products, c_lo t, the tail,
    // (c_hi / 2) (t^2).lo and (c_lo / 2) t^2
    const float small = add(add(sub(a.lo, q.lo), fma(w, kInvLn2Lo, tail)),
                            -fma(mul(0.5f, kInvLn2Hi), sq.lo, mul(mul(0.5f, kInvLn2Lo), sq.hi)));
    const F2 l1 = fast_two_sum(a.hi, -q.hi);              // |q.hi| < |a.hi| / 256
    const F2 lt = fast_two_sum(l1.hi, add(l1.lo, small)); // log2(1 + t)
    const F2 frac = add2(F2{en.nl_hi, en.nl_lo}, lt);      // log2 u, in [0, 1)
    const F2 whole = two_sum((float)(ex - 127), frac.hi);
    return two_sum(whole.hi, add(whole.lo, frac.lo));
}

// 2^z for a double-float z as 2^n (m.hi + m.lo), with m.hi + m.lo in about
// [0.7, 1.42] not yet rounded: the caller rounds m once and scales it by 2^n.
// z.hi is a multiple of a power of two g <= 1/32 with |z.lo| <= g / 2 (a
// normalized pair with |z.hi| < 2^19, or one whose high part had an integer
// subtracted): then z.hi - n and z.hi - n - j/32 are exact multiples of g, so
// the low part joins them in one FastTwoSum.
COAT_HD F2 exp2_df_parts(F2 z, const Tables& t, int& n_out) {
    const float n = rint(z.hi);
    const float fh = sub(z.hi, n);                 // exact, |fh| <= 0.5
    const float jf = rint(mul(fh, 32.0f));         // -16..16
    // clamped so that no input (even a non-finite one) can index outside the
    // 33-entry table
    const int j0 = (int)jf;
    const int j = j0 < -16 ? -16 : (j0 > 16 ? 16 : j0);
    const F2 r = fast_two_sum(sub(fh, mul(jf, 0.03125f)), z.lo);   // |r| <= 1/64 + |z.lo|
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
