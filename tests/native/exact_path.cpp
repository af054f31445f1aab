// The step kernel's exact path run on the host: the same double-float code and
// tables (IEEE-exact operations only, so the host reproduces the device), with
// the certain-rounding test and the float64 recomputation of the rare values
// it cannot round with certainty.
//
// Reads lines from stdin, one case per line, and prints one result line each:
//   "d code S_bits k_bits"   -> "prev_bits slow"   the dequantized magnitude
//                                                 (|E4M3(code)| S)^(1/k), fp32
//   "k mx_bits mn_bits"      -> "k_bits slow"      the group exponent for the
//                                                 extremes mx >= mn > 0
// slow = 1 when the float64 recomputation decided the value.
#include <cstdio>
#include <cstring>

#define COAT_CONST
#include "coat_tables.inc"
#include "coat_round.cuh"

using coat::df::F2;

static float u2f(unsigned u) { float f; std::memcpy(&f, &u, 4); return f; }
static unsigned f2u(float f) { unsigned u; std::memcpy(&u, &f, 4); return u; }
static F2 cdf(const unsigned* p) { return F2{u2f(p[0]), u2f(p[1])}; }

// |E4M3| of a magnitude code (bias 7, subnormal below 8), as the kernel forms it
static float e4m3_mag(unsigned mag) {
    if (mag >= 8u) return u2f((((mag >> 3) + 120u) << 23) | ((mag & 7u) << 20));
    return (float)mag * 0.001953125f;
}

int main() {
    static coat::df::LogEntry logr[256];
    float e_hi[33], e_lo[33];
    std::memcpy(logr, kLog2Recip, sizeof(logr));
    for (int i = 0; i < 33; ++i) { e_hi[i] = u2f(kExp2FracHi[i]); e_lo[i] = u2f(kExp2FracLo[i]); }
    const coat::df::Tables t{logr, e_hi, e_lo};
    const coat::df::KConsts kc{cdf(kLog2RDf), cdf(kGuardLoDf), cdf(kGuardHiDf),
                               u2f(kLog2RRcp), u2f(kGuardLoRcp), u2f(kGuardHiRcp), 8.0f,
                               448.0 * 512.0, -125.0, 126.0};
    char kind[4];
    unsigned a = 0, b = 0, c = 0;
    while (std::scanf("%3s", kind) == 1) {
        if (kind[0] == 'd') {
            if (std::scanf("%u %u %u", &a, &b, &c) != 3) return 2;
            const unsigned mag = a & 0x7Fu;
            const float S = u2f(b), k = u2f(c);
            const F2 rkd = coat::df::recip21(k);
            const F2 A = coat::df::add2(coat::df::log2_df(S, t), cdf(kLog2_448Df));
            const F2 L = {u2f(kLog2Frac448Hi[mag]), u2f(kLog2Frac448Lo[mag])};
            bool slow = false;
            float prev;
            if (rkd.hi == 1.0f && rkd.lo == 0.0f) {
                prev = e4m3_mag(mag) * S;           // k = 1: one correctly rounded product
            } else {
                prev = coat::df::dequant_certain(L, A, rkd, e4m3_mag(mag), S, k, t, slow);
            }
            std::printf("%u %d\n", f2u(prev), slow ? 1 : 0);
        } else if (kind[0] == 'k') {
            if (std::scanf("%u %u", &a, &b) != 2) return 2;
            const float mx = u2f(a), mn = u2f(b);
            const F2 Lmx = coat::df::log2_df(mx, t);
            const F2 Lmn = mn < mx ? coat::df::log2_df(mn, t) : Lmx;
            bool slow = false;
            const float k = coat::df::k_certain(mx, mn, Lmx, Lmn, kc, slow);
            std::printf("%u %d\n", f2u(k), slow ? 1 : 0);
        } else {
            return 2;
        }
    }
    return 0;
}
