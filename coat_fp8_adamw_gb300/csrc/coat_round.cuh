// coat_round.cuh -- fp32 rounding with certainty for values computed in
// double-float, and the float64 recomputations for the rare values that
// cannot be rounded with certainty.
//
// The exact path of the step rounds a double-float approximation of each
// value to fp32 once.  That equals the correctly rounded value unless the
// exact value lies nearer than the approximation's error to an fp32 rounding
// midpoint.  For a group's extreme moments such a one-ulp slip matters: when
// the smallest |m_t| of a group is the remainder of a partial cancellation, a
// one-ulp change of the dequantized previous moment is many ulps of m_t, and
// through k it moves S by several 1e-6 (COAT review page, section 3: S and
// k follow from the group's max and min).  Ziv's rounding test decides, from
// the approximation and its error bound, whether the rounding is certain;
// the few values where it is not are recomputed in float64 from the same
// definitions the method states.
#pragma once

#include <cmath>

#include "coat_df.cuh"

#if defined(__CUDACC__)
#define COAT_HD_OUTLINE static __host__ __device__ __noinline__
#else
#define COAT_HD_OUTLINE static inline
#endif

namespace coat {
namespace df {

COAT_HD float abs1(float x) { return from_bits(bits(x) & 0x7FFFFFFFu); }

// RN(v) for a double-float v = hi + lo (|lo| <= |hi|) that lies within a
// relative distance eps of an exact value x.  `certain` is true when RN(x)
// must equal RN(v): no fp32 rounding midpoint lies within eps |v| of v.  The
// nearest midpoint is half an ulp from RN(v) on the side of the remainder
// v - RN(v); at a power of two the ulp below is half the ulp above.
COAT_HD float round_certain(F2 v, float eps, bool& certain) {
    const F2 s = fast_two_sum(v.hi, v.lo);   // s.hi = RN(v), s.lo = v - s.hi exactly
    const float r = s.hi;
    if (r == 0.0f) {
        certain = v.lo == 0.0f;
        return r;
    }
    const uint32_t b = bits(r);
    const bool outward = (s.lo > 0.0f) == (r > 0.0f);   // remainder points away from zero
    const float nb = from_bits(outward ? b + 1u : b - 1u);
    const float half = mul(0.5f, abs1(sub(nb, r)));    // exact: a power of two
    const float d = sub(half, abs1(s.lo));             // distance to that midpoint
    certain = d > mul(eps, abs1(r));
    return r;
}
// The same test with the relative error bound given as num / den (den > 0):
// d > (num / den) |r| taken as d den > num |r|, without the division (the two
// products' roundings move the bound by a relative 2^-23, far inside its
// margin).
COAT_HD float round_certain_q(F2 v, float num, float den, bool& certain) {
    const F2 s = fast_two_sum(v.hi, v.lo);
    const float r = s.hi;
    if (r == 0.0f) {
        certain = v.lo == 0.0f;
        return r;
    }
    const uint32_t b = bits(r);
    const bool outward = (s.lo > 0.0f) == (r > 0.0f);
    const float nb = from_bits(outward ? b + 1u : b - 1u);
    const float half = mul(0.5f, abs1(sub(nb, r)));
    const float d = sub(half, abs1(s.lo));
    certain = mul(d, den) > mul(num, abs1(r));
    return r;
}

// The dequantized moment sign-free: (|E4M3(q)| S)^(1/k) in float64, rounded
// once to fp32 (the definition, for the values the double-float path cannot
// round with certainty).  `mag` is the code's magnitude value; S > 0, k > 0.
COAT_HD_OUTLINE float dequant_f64(float mag, float S, float k) {
    return (float)pow((double)mag * (double)S, 1.0 / (double)k);
}

// k of a group from its extremes mx >= mn > 0 in float64, rounded once to
// fp32: min(log R / log(mx / mn), cap), then lowered so that S = mx^k / 448
// stays inside [2^s_lo, 2^s_hi] (the readings of the method's open points:
// the exponent formula, a cap, and the S-range guard).  mn == mx gives k = 1
// before the guard.
COAT_HD_OUTLINE float k_f64(float mx, float mn, double R, double cap, double s_lo, double s_hi) {
    double k = 1.0;
    if (mn < mx) {
        k = log(R) / log((double)mx / (double)mn);
        k = k < cap ? k : cap;
    }
    const double l = log2((double)mx), l448 = log2(448.0);
    if (l < 0.0) {
        const double bound = (l448 + s_lo) / l;
        k = bound < k ? bound : k;
    } else if (l > 0.0) {
        const double bound = (l448 + s_hi) / l;
        k = bound < k ? bound : k;
    }
    return (float)k;
}

// Relative error bounds of the double-float values that the two functions
// below round, with a factor 4 of margin over the largest errors measured
// against long double on 2 x 10^7 random inputs each:
//  - the dequantized moment 2^z, z = (L + A) / k: within
//    2^-44.2 (|z| + |A| / k + 1) (log2 of 448 S and the product with 1/k carry
//    absolute errors proportional to their size, exp2 adds ~2^-47);
//  - k = log2 R / (log2 max - log2 min): within
//    2^-45.2 (2 + |log2 max| + |log2 min|) / |log2 max - log2 min|.
COAT_HD float dequant_err_bound(float z_abs, float A_abs, float rk) {
    return mul(0x1p-42f, add(add(z_abs, mul(A_abs, rk)), 1.0f));
}
COAT_HD float k_err_num(float lmx_abs, float lmn_abs) {
    return mul(0x1p-43f, add(add(2.0f, lmx_abs), lmn_abs));
}
COAT_HD float k_err_bound(float lmx_abs, float lmn_abs, float d_abs) {
    return div(k_err_num(lmx_abs, lmn_abs), d_abs);
}

// Correctly rounded fp32 magnitude of a dequantized moment
// (|E4M3(q)| S)^(1/k), from L = log2(|E4M3(q)| / 448), A = log2(448 S) and
// 1/k as double-floats: 2^((L + A) / k) rounded once when that rounding is
// certain, else (rarely) the float64 definition.  A result in the fp32
// subnormal range (scaling it would round twice) also takes the float64 path.
// `mag` is |E4M3(q)| (> 0), S > 0, k the stored exponent; `slow` reports the
// float64 path.  dequant_try is the first part alone: the double-float value
// rounded once, with `slow` set where the caller must take the float64 path.
COAT_HD float dequant_try(F2 L, F2 A, F2 rkd, const Tables& t, bool& slow) {
    const F2 z = mul22(add2(L, A), rkd);
    int n = 0;
    const F2 m = exp2_df_parts(z, t, n);
    bool certain = false;
    const float r = round_certain(m, dequant_err_bound(abs1(z.hi), abs1(A.hi), rkd.hi), certain);
    const float x = scale2(r, n);
    slow = !certain || !(x >= 1.17549435e-38f);
    return x;
}
COAT_HD float dequant_certain(F2 L, F2 A, F2 rkd, float mag, float S, float k, const Tables& t,
                              bool& slow) {
    const float x = dequant_try(L, A, rkd, t, slow);
    return slow ? dequant_f64(mag, S, k) : x;
}

// The constants of the exponent rule: log2 R, the cap, the guard numerators
// log2 448 - 125 and log2 448 + 126 (double-floats), and R with the S range
// for the float64 recomputation.
struct KConsts {
    F2 log2R, guard_lo, guard_hi;
    float rcp_log2R, rcp_guard_lo, rcp_guard_hi;   // 1 / the high parts
    float cap;
    double R, s_lo, s_hi;
};

// k of a group from its extremes mx >= mn > 0 (mn = mx: one magnitude) and
// their double-float log2: min(log2 R / (log2 mx - log2 mn), cap), lowered by
// the S-range guard, every candidate rounded once to fp32.  The minimum of
// correctly rounded candidates is the correctly rounded minimum, so the
// result is exact unless a candidate that could be the minimum has an
// uncertain rounding; then the float64 definition decides (`slow`).
COAT_HD float k_certain(float mx, float mn, F2 Lmx, F2 Lmn, const KConsts& c, bool& slow) {
    float k = 1.0f;
    float doubt = 3.4e38f;        // smallest uncertain candidate
    if (mn > 0.0f && mn < mx) {
        const F2 D = add2(Lmx, neg2(Lmn));
        bool certain = false;
        const float kf = round_certain_q(div22_parts_k(c.log2R, c.rcp_log2R, D),
                                         k_err_num(abs1(Lmx.hi), abs1(Lmn.hi)), abs1(D.hi), certain);
        if (!certain) doubt = kf;
        k = kf < c.cap ? kf : c.cap;
    }
    if (Lmx.hi != 0.0f) {
        bool certain = false;
        const bool neg = Lmx.hi < 0.0f;
        const float kg = round_certain_q(div22_parts_k(neg ? c.guard_lo : c.guard_hi,
                                                       neg ? c.rcp_guard_lo : c.rcp_guard_hi, Lmx),
                                         k_err_num(abs1(Lmx.hi), 0.0f), abs1(Lmx.hi), certain);
        if (!certain && kg < doubt) doubt = kg;
        k = kg < k ? kg : k;
    }
    // an uncertain candidate more than a few ulps above the minimum cannot
    // become it (its error bound is far below an ulp)
    slow = doubt <= mul(k, 1.0000005f);
    return slow ? k_f64(mx, mn, c.R, (double)c.cap, c.s_lo, c.s_hi) : k;
}

}  // namespace df
}  // namespace coat
