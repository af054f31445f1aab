// Host-side check of coat_round.cuh: round_certain never reports a rounding
// as certain when the exact value rounds differently, also for values placed
// right at fp32 rounding midpoints, and reports uncertainty rarely otherwise.
// The float64 recomputations are compared with libm on the same definitions.
// Prints one line of key=value statistics; tests/test_round_host.py asserts.
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <random>

#include "coat_round.cuh"

using coat::df::F2;

static F2 split(double v) {
    const float hi = (float)v;
    return F2{hi, (float)(v - (double)hi)};
}

int main() {
    std::mt19937_64 rng(4242);
    std::uniform_real_distribution<double> U(0.0, 1.0);
    const float eps = 0x1p-40f;
    long wrong = 0, random_uncertain = 0, random_n = 0, near_n = 0, near_certain_wrong = 0,
         near_uncertain = 0;
    // random exact values x, approximations within eps/2 of x (the double-float
    // split adds at most 2^-48 more)
    for (int i = 0; i < 4000000; ++i) {
        const double x = std::exp2(-60.0 + 70.0 * U(rng)) * (U(rng) < 0.5 ? -1.0 : 1.0);
        const double v = x * (1.0 + (U(rng) - 0.5) * (double)eps);
        bool certain = false;
        const float r = coat::df::round_certain(split(v), eps, certain);
        ++random_n;
        if (!certain) ++random_uncertain;
        else if (r != (float)x) ++wrong;
    }
    // exact values at and around fp32 midpoints: x = midpoint * (1 + t),
    // |t| from 0 to a few eps, approximation anywhere within eps of x
    for (int i = 0; i < 4000000; ++i) {
        const float a = (float)std::exp2(-60.0 + 70.0 * U(rng));
        const float b = std::nextafter(a, 2.0f * a);
        const double mid = 0.5 * ((double)a + (double)b);     // exact in double
        const double t = (U(rng) - 0.5) * 6.0 * (double)eps;
        const double x = mid * (1.0 + t);
        const double v = x * (1.0 + (U(rng) - 0.5) * 1.9 * (double)eps);
        bool certain = false;
        const float r = coat::df::round_certain(split(v), eps, certain);
        ++near_n;
        if (!certain) ++near_uncertain;
        else if (r != (float)x) ++near_certain_wrong;
    }
    // the ratio form (bound num / den, compared without a division) at and
    // around midpoints, den spread over the range the exponent rule gives
    long q_wrong = 0, q_uncertain = 0;
    for (int i = 0; i < 2000000; ++i) {
        const float a = (float)std::exp2(-60.0 + 70.0 * U(rng));
        const float b = std::nextafter(a, 2.0f * a);
        const double mid = 0.5 * ((double)a + (double)b);
        const float den = (float)std::exp2(-3.0 + 12.0 * U(rng));
        const float num = eps * den;
        const double t = (U(rng) - 0.5) * 6.0 * (double)eps;
        const double x = mid * (1.0 + t);
        const double v = x * (1.0 + (U(rng) - 0.5) * 1.9 * (double)eps);
        bool certain = false;
        const float r = coat::df::round_certain_q(split(v), num, den, certain);
        if (!certain) ++q_uncertain;
        else if (r != (float)x) ++q_wrong;
    }
    // the float64 recomputations against libm on the same formulas
    long dq_diff = 0, k_diff = 0;
    for (int i = 0; i < 100000; ++i) {
        const float mag = (float)std::exp2(std::floor(18.0 * U(rng)) - 9.0) * (1.0f + (float)std::floor(8.0 * U(rng)) / 8.0f);
        const float S = (float)std::exp2(-100.0 * U(rng));
        const float k = (float)(0.6 + 7.4 * U(rng));
        const float want = (float)std::pow((double)mag * (double)S, 1.0 / (double)k);
        if (coat::df::dequant_f64(mag, S, k) != want) ++dq_diff;
        const float mx = (float)std::exp2(-40.0 * U(rng)), mn = mx * (float)std::exp2(-30.0 * U(rng));
        double kk = std::log(229376.0) / std::log((double)mx / (double)mn);
        kk = kk < 8.0 ? kk : 8.0;
        const double l = std::log2((double)mx);
        if (l < 0.0 && (std::log2(448.0) - 125.0) / l < kk) kk = (std::log2(448.0) - 125.0) / l;
        if (coat::df::k_f64(mx, mn, 229376.0, 8.0, -125.0, 126.0) != (float)kk) ++k_diff;
    }
    std::printf("random_wrong=%ld random_uncertain_frac=%.3e near_n=%ld near_certain_wrong=%ld "
                "near_uncertain_frac=%.3e dequant_diff=%ld k_diff=%ld q_wrong=%ld q_uncertain_frac=%.3e\n",
                wrong, (double)random_uncertain / random_n, near_n, near_certain_wrong,
                (double)near_uncertain / near_n, dq_diff, k_diff, q_wrong, (double)q_uncertain / 2000000);
    return 0;
}
