// Host-side check of the double-float toolkit used by the kernels
// (coat_fp8_adamw_gb300/csrc/coat_df.cuh) against float64 libm.
// Prints one line of key=value statistics; tests/test_df_host.py asserts on them.
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <random>

#define COAT_CONST
#include "coat_df.cuh"
#include "coat_tables.inc"

using coat::df::F2;

static float u2f(unsigned u) { float f; std::memcpy(&f, &u, 4); return f; }

int main() {
    float lc_hi[64], lc_lo[64], e_hi[33], e_lo[33];
    for (int i = 0; i < 64; ++i) { lc_hi[i] = u2f(kLog2CenterHi[i]); lc_lo[i] = u2f(kLog2CenterLo[i]); }
    for (int i = 0; i < 33; ++i) { e_hi[i] = u2f(kExp2FracHi[i]); e_lo[i] = u2f(kExp2FracLo[i]); }
    coat::df::Tables t{lc_hi, lc_lo, e_hi, e_lo};
    std::mt19937_64 rng(12345);
    std::uniform_real_distribution<double> U(0.0, 1.0);

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
                "div_miss_frac=%.3e dot_miss_frac=%.3e\n",
                log2_max_abs, log2_max_near1, (double)exp2_miss / exp2_n, exp2_max_rel,
                (double)div_miss / N, (double)dot_miss / N);
    return 0;
}
