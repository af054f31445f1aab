// The step kernel's exact dequantization of one stored moment, run on the host
// with the same double-float code and tables (IEEE-exact operations only, so
// the host reproduces the device): A = log2(448 S) and 1/k in double-float,
// then 2^((L(q) + A)/k) rounded once to fp32.  Reads "code S_bits k_bits" from
// argv, prints the result's bits.
#include <cstdio>
#include <cstdlib>
#include <cstring>

#define COAT_CONST
#include "coat_df.cuh"
#include "coat_tables.inc"

using coat::df::F2;

static float u2f(unsigned u) { float f; std::memcpy(&f, &u, 4); return f; }

int main(int argc, char** argv) {
    if (argc != 4) return 2;
    const unsigned code = (unsigned)std::strtoul(argv[1], nullptr, 10);
    const float S = u2f((unsigned)std::strtoul(argv[2], nullptr, 10));
    const float k = u2f((unsigned)std::strtoul(argv[3], nullptr, 10));
    float lc_hi[64], lc_lo[64], e_hi[33], e_lo[33];
    for (int i = 0; i < 64; ++i) { lc_hi[i] = u2f(kLog2CenterHi[i]); lc_lo[i] = u2f(kLog2CenterLo[i]); }
    for (int i = 0; i < 33; ++i) { e_hi[i] = u2f(kExp2FracHi[i]); e_lo[i] = u2f(kExp2FracLo[i]); }
    const coat::df::Tables t{lc_hi, lc_lo, e_hi, e_lo};
    const unsigned mag = code & 0x7Fu;
    const F2 rkd = coat::df::div21(F2{1.0f, 0.0f}, k);
    const F2 A = coat::df::add2(coat::df::log2_df(S, t), F2{u2f(kLog2_448Df[0]), u2f(kLog2_448Df[1])});
    const F2 L = {u2f(kLog2Frac448Hi[mag]), u2f(kLog2Frac448Lo[mag])};
    const float prev = coat::df::exp2_df(coat::df::mul22(coat::df::add2(L, A), rkd), t);
    unsigned u;
    std::memcpy(&u, &prev, 4);
    std::printf("%u\n", u);
    return 0;
}
