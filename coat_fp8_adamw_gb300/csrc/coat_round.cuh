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
#define COAT_HD_OUTLINE __host__ __device__ __noinline__
#else
#define COAT_HD_OUTLINE inline
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

}  // namespace df
}  // namespace coat
