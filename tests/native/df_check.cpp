// Host-side check of the double-float toolkit used by the kernels
// (coat_fp8_adamw_gb300/csrc/coat_df.cuh) against float64 libm and long
// double, and of the error bounds that the certain-rounding test relies on.
// Prints one line of key=value statistics; tests/test_df_host.py asserts on them.
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <random>

#define COAT_CONST
#include "coat_tables.inc"
#include "coat_round.cuh"

using coat::df::F2;

static float u2f(unsigned u) { float f; std::memcpy(&f, &u, 4); return f; }
static F2 cdf(const unsigned* p) { return F2{u2f(p[0]), u2f(p[1])}; }

int main() {
    static coat::df::LogEntry logr[256];
    float e_hi[33], e_lo[33];
    std::memcpy(logr, kLog2Recip, sizeof(logr));
    for (int i = 0; i < 33; ++i) { e_hi[i] = u2f(kExp2FracHi[i]); e_lo[i] = u2f(kExp2FracLo[i]); }
    coat::df::Tables t{logr, e_hi, e_lo};
    std::mt19937_64 rng(12345);
    std::uniform_real_distribution<double> U(0.0, 1.0);

    // the log2 reduction: for every fp32 significand u, fma(u, r_j, -1) in
    // fp32 equals u r_j - 1 (exact in float64: 24 + 9 significant bits), with
    // r_j as the kernels form it
    long reduce_inexact = 0;
    double reduce_max = 0;
    for (unsigned m = 0; m < (1u << 23); ++m) {
        const float u = u2f(0x3F800000u | m);
        const float r = coat::df::log_recip(m >> 15);
        const double exact = (double)u * (double)r - 1.0;
        if ((double)std::fma(u, r, -1.0f) != exact) ++reduce_inexact;
        if (std::fabs(exact) > reduce_max) reduce_max = std::fabs(exact);
    }
    // log2 of every significand u in [1, 2) against long double: a table entry
    // that does not belong to the kernels' r_j would be off by ~2^-9
    double log2_sig_max_abs = 0;
    for (unsigned m = 0; m < (1u << 23); ++m) {
        const float u = u2f(0x3F800000u | m);
        const F2 r = coat::df::log2_df(u, t);
        const double err = (double)fabsl(((long double)r.hi + (long double)r.lo) - log2l((long double)u));
        if (err > log2_sig_max_abs) log2_sig_max_abs = err;
    }
    // log2 against long double: the largest error over the stated bound
    // 2^-46 + 2^-47 |log2 x|
    double log2_bound_ratio = 0;
    for (int i = 0; i < 4000000; ++i) {
        float x = (float)std::exp2(-149.0 + 277.0 * U(rng));
        if (i % 3 == 0) x = (float)(1.0 + (U(rng) - 0.5) * 0.03);
        if (!(x > 0) || !std::isfinite(x)) continue;
        const F2 r = coat::df::log2_df(x, t);
        const long double want = log2l((long double)x);
        const double err = (double)fabsl(((long double)r.hi + (long double)r.lo) - want);
        const double bound = std::ldexp(1.0, -46) + std::ldexp(1.0, -47) * std::fabs((double)want);
        if (err / bound > log2_bound_ratio) log2_bound_ratio = err / bound;
    }
    // the error bounds of the certain-rounding test (coat_round.cuh): the
    // largest relative error of the double-float dequantized moment (before
    // its one rounding) and of the double-float k quotient, each over its
    // bound, against long double
    const F2 l448 = cdf(kLog2_448Df), l2R = cdf(kLog2RDf);
    double dequant_bound_ratio = 0, k_bound_ratio = 0;
    for (int i = 0; i < 2000000; ++i) {
        const int code = 1 + (int)(125 * U(rng));
        const float S = (float)std::exp2(-120.0 + 130.0 * U(rng));
        const float k = (float)(1.0 + 7.0 * U(rng));
        const F2 rkd = coat::df::recip21(k);
        const F2 A = coat::df::add2(coat::df::log2_df(S, t), l448);
        const F2 L = {u2f(kLog2Frac448Hi[code]), u2f(kLog2Frac448Lo[code])};
        const F2 z = coat::df::mul22(coat::df::add2(L, A), rkd);
        int n = 0;
        const F2 m = coat::df::exp2_df_parts(z, t, n);
        const long double want = powl(2.0L, ((long double)L.hi + (long double)L.lo + log2l((long double)S) +
                                             log2l(448.0L)) / (long double)k - (long double)n);
        const double rel = (double)fabsl(((long double)m.hi + (long double)m.lo) / want - 1.0L);
        const double b = coat::df::dequant_err_bound(std::fabs(z.hi), std::fabs(A.hi), rkd.hi);
        if (rel / b > dequant_bound_ratio) dequant_bound_ratio = rel / b;

        const float mxv = (float)std::exp2(-100.0 + 120.0 * U(rng));
        const float mnv = (float)((double)mxv * std::exp2(-(0.5 + 40.0 * U(rng))));
        if (!(mnv > 0)) continue;
        const F2 Lmx = coat::df::log2_df(mxv, t), Lmn = coat::df::log2_df(mnv, t);
        const F2 D = coat::df::add2(Lmx, coat::df::neg2(Lmn));
        const F2 q = coat::df::div22_parts_k(l2R, u2f(kLog2RRcp), D);
        const long double kw = log2l(448.0L * 512.0L) / (log2l((long double)mxv) - log2l((long double)mnv));
        const double krel = (double)fabsl(((long double)q.hi + (long double)q.lo) / kw - 1.0L);
        const double kb = coat::df::k_err_bound(std::fabs(Lmx.hi), std::fabs(Lmn.hi), std::fabs(D.hi));
        if (krel / kb > k_bound_ratio) k_bound_ratio = krel / kb;
    }
    // x 2^n against ldexp rounded once to fp32, for every n in [-260, 260]
    // (the one-factor path, the two-factor path, subnormal results, overflow)
    long scale2_miss = 0;
    for (int i = 0; i < 2000; ++i) {
        const float x = (float)(0.5 + 1.5 * U(rng)) * (i & 1 ? -1.0f : 1.0f);
        for (int n = -260; n <= 260; ++n) {
            const float want = (float)std::ldexp((double)x, n < -252 ? -252 : (n > 254 ? 254 : n));
            if (coat::df::scale2(x, n) != want) ++scale2_miss;
        }
    }
    // log2: absolute error of hi+lo against libm log2 in double
    double log2_max_abs = 0, log2_max_near1 = 0;
    const int N = 2000000;
    for (int i = 0; i < N; ++i) {
        double l = -149.0 + 277.0 * U(rng);
        float x = (float)std::exp2(l);
        if (!(x > 0) || !std::isfinite(x)) continue;
        if (i % 7 == 0) x = 1.0f + (float)((U(rng) - 0.5) * 1e-3);  // near 1
        F2 r = coat::df::log2_df(x, t);
        double err = std::fabs(((double)r.hi + (double)r.lo) - std::log2((double)x));
        if (i % 7 == 0) { if (err > log2_max_near1) log2_max_near1 = err; }
        else if (err > log2_max_abs) log2_max_abs = err;
    }
    // exp2: fraction of results that differ from the correctly rounded value
    long exp2_miss = 0, exp2_n = 0;
    double exp2_max_rel = 0;
    for (int i = 0; i < N; ++i) {
        double z = -125.0 + 251.0 * U(rng);
        float hi = (float)z;
        float lo = (float)(z - (double)hi);
        double zz = (double)hi + (double)lo;
        float want = (float)std::exp2(zz);
        float got = coat::df::exp2_df(F2{hi, lo}, t);
        exp2_n++;
        if (got != want) exp2_miss++;
        double rel = std::fabs((double)got / std::exp2(zz) - 1.0);
        if (rel > exp2_max_rel) exp2_max_rel = rel;
    }
    // division of double-floats rounded once
    long div_miss = 0;
    for (int i = 0; i < N; ++i) {
        double a = std::exp2(40.0 * (U(rng) - 0.5)), b = std::exp2(40.0 * (U(rng) - 0.5));
        float ah = (float)a, al = (float)(a - ah), bh = (float)b, bl = (float)(b - bh);
        double q = ((double)ah + (double)al) / ((double)bh + (double)bl);
        if (coat::df::div22_rn(F2{ah, al}, F2{bh, bl}) != (float)q) div_miss++;
    }
    // a*b + c*d rounded once
    long dot_miss = 0;
    for (int i = 0; i < N; ++i) {
        float a = (float)(U(rng) * 2 - 1), b = (float)U(rng), c = (float)(U(rng) * 2 - 1),
              d = (float)(U(rng) * 1e-3);
        double ex = (double)a * b + (double)c * d;
        if (coat::df::dot2_rn(a, b, c, d) != (float)ex) dot_miss++;
    }
    std::printf("log2_max_abs=%.3e log2_max_abs_near1=%.3e exp2_miss_frac=%.3e exp2_max_rel=%.3e "
                "div_miss_frac=%.3e dot_miss_frac=%.3e reduce_inexact=%ld reduce_max=%.6e "
                "log2_bound_ratio=%.4f dequant_bound_ratio=%.4f k_bound_ratio=%.4f log2_sig_max_abs=%.3e "
                "scale2_miss=%ld\n",
                log2_max_abs, log2_max_near1, (double)exp2_miss / exp2_n, exp2_max_rel,
                (double)div_miss / N, (double)dot_miss / N, reduce_inexact, reduce_max,
                log2_bound_ratio, dequant_bound_ratio, k_bound_ratio, log2_sig_max_abs, scale2_miss);
    return 0;
}
