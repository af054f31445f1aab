// coat_device.cuh -- device-side building blocks shared by the GB300 kernels:
// FP8 E4M3 packing, base-2 exp/log through the SFU, per-group Dynamic Range
// Expansion parameters, and the 128-bit streaming loads/stores.
//
// Method: COAT paper-review page (xllm-io), section 3 core formulas --
//   FP8 quantization  X_FP8 = round(X / S), S = max|X| / 448
//   expansion         f(x) = sign(x)|x|^k, R_X = max|X| / min|X|,
//                     k = log_{R_X}(R_E4M3)
// with the library's readings: min over non-zero |x|, k <= 8, S kept in
// [2^-125, 2^126], R_E4M3 = 448 / 2^-9, round-to-nearest-even saturating
// encoding.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#define COAT_CONST __constant__
#include "coat_tables.inc"
#include "coat_df.cuh"
#include "coat_round.cuh"

namespace coat {

// The same tables in global memory: filling shared-memory copies from these
// is one coalesced load per warp, where reading constant memory with a
// different index in every lane serializes the warp.
namespace gtab {
#undef COAT_CONST
#define COAT_CONST __device__
#include "coat_tables.inc"
#undef COAT_CONST
#define COAT_CONST __constant__
}  // namespace gtab

constexpr int kVec = 16;         // elements per thread: one 128-bit load of codes
constexpr int kThreads = 256;    // threads per CTA

// log2(448), log2(R_E4M3) = log2(448 * 2^9), the k cap, and the S-range guard
// numerators (log2 448 - 125, log2 448 + 126), as float constants.
constexpr float kLog2_448 = 8.8073549220576041f;
constexpr float kLog2R = 17.807354922057604f;
constexpr float kKCap = 8.0f;
constexpr float kGuardLo = 8.8073549220576041f - 125.0f;
constexpr float kGuardHi = 8.8073549220576041f + 126.0f;

// ---------------------------------------------------------------------------
// SFU approximations, as documented PTX instructions.  The .ftz forms are one
// SFU instruction each; they flush subnormal inputs and results to zero,
// which only touches values below 2^-126 (documented at each use).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float ex2_ftz(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float lg2_ftz(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp_ftz(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float sqrt_ftz(float x) {
    float y;
    asm("sqrt.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float lg2_approx(float x) {
    float y;
    asm("lg2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Packed fp32 pairs (PTX .f32x2): each half rounds like the scalar instruction.
__device__ __forceinline__ uint64_t pk(float x, float y) {
    uint64_t u;
    asm("mov.b64 %0, {%1, %2};" : "=l"(u) : "f"(x), "f"(y));
    return u;
}
__device__ __forceinline__ void upk(uint64_t u, float& x, float& y) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(x), "=f"(y) : "l"(u));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Two fp32 values -> two E4M3 codes (round to nearest even, saturate to
// +-448), packed little-endian: lo -> bits 0..7, hi -> bits 8..15.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return (uint32_t)r;
}

// ---------------------------------------------------------------------------
// 128-bit streaming memory access (evict-first: the data set exceeds L2)
// ---------------------------------------------------------------------------
__device__ __forceinline__ float4 ld_cs(const float4* p) { return __ldcs(p); }
__device__ __forceinline__ uint4 ld_cs(const uint4* p) { return __ldcs(p); }
__device__ __forceinline__ void st_cs(float4* p, float4 v) { __stcs(p, v); }
__device__ __forceinline__ void st_cs(uint4* p, uint4 v) { __stcs(p, v); }

// Fresh per-group parameters from the group's max and smallest non-zero
// magnitude (section 3: R_X = max/min, k = log_{R_X} R_E4M3, S = max|f(X)|/448
// = max^k / 448), with the library's cap and S-range guard.
struct QuantParams {
    float k;
    float S;
    float inv_mx;  // 1/max (0 for an all-zero group)
};

// Shared-memory copy of the double-float tables (divergent indices: constant
// memory would serialize them).
struct SmemTables {
    df::LogEntry logr[256];
    float exp2j_hi[33], exp2j_lo[33];
};

__device__ __forceinline__ void load_smem_tables(SmemTables& st, int tid, int nthreads) {
    const uint2* src = reinterpret_cast<const uint2*>(gtab::kLog2Recip);
    for (int i = tid; i < 256; i += nthreads) reinterpret_cast<uint2*>(st.logr)[i] = src[i];
    for (int i = tid; i < 33; i += nthreads) {
        st.exp2j_hi[i] = __uint_as_float(gtab::kExp2FracHi[i]);
        st.exp2j_lo[i] = __uint_as_float(gtab::kExp2FracLo[i]);
    }
}

__device__ __forceinline__ df::Tables tables_of(const SmemTables& st) {
    return df::Tables{st.logr, st.exp2j_hi, st.exp2j_lo};
}

__device__ __forceinline__ df::F2 const_df(const unsigned int* p) {
    return df::F2{__uint_as_float(p[0]), __uint_as_float(p[1])};
}

// The exponent rule's constants (R_E4M3 = 448 / 2^-9, cap 8, S kept in
// [2^-125, 2^126]) for df::k_certain.
__device__ __forceinline__ df::KConsts k_consts() {
    return df::KConsts{const_df(kLog2RDf), const_df(kGuardLoDf), const_df(kGuardHiDf),
                       __uint_as_float(kLog2RRcp), __uint_as_float(kGuardLoRcp), __uint_as_float(kGuardHiRcp),
                       kKCap, 448.0 * 512.0, -125.0, 126.0};
}

// Fresh per-group parameters with k correctly rounded to fp32 (double-float
// logs and quotient, rounded once when that is certain, float64 otherwise)
// and S = 2^(k log2 max - log2 448) rounded once.
// quant_params_logs takes the two logs formed by the caller: Lmx = log2 mx,
// Lmn = log2 mn (or Lmx when mn is zero or not below mx).
__device__ __forceinline__ QuantParams quant_params_logs(float mx, float mn, df::F2 Lmx, df::F2 Lmn,
                                                         const df::Tables& t) {
    QuantParams q;
    if (!(mx > 0.0f)) {
        q.k = 1.0f;
        q.S = 0.0f;
        q.inv_mx = 0.0f;
        return q;
    }
    bool slow = false;
    const float k = df::k_certain(mx, mn, Lmx, Lmn, k_consts(), slow);
    const df::F2 e = df::add2(df::mul21(Lmx, k), df::neg2(const_df(kLog2_448Df)));
    q.k = k;
    q.S = df::exp2_df(e, t);
    q.inv_mx = __frcp_rn(mx);
    return q;
}
__device__ __forceinline__ QuantParams quant_params_precise(float mx, float mn,
                                                            const df::Tables& t) {
    if (!(mx > 0.0f)) return quant_params_logs(mx, mn, df::F2{0.0f, 0.0f}, df::F2{0.0f, 0.0f}, t);
    const df::F2 Lmx = df::log2_df(mx, t);
    const df::F2 Lmn = (mn > 0.0f && mn < mx) ? df::log2_df(mn, t) : Lmx;
    return quant_params_logs(mx, mn, Lmx, Lmn, t);
}

// Scaled, expanded value y = 448 sign(x) (|x| / max)^k, ready for E4M3 rounding.
// `r` is |x| / max (computed by the caller), `x` supplies the sign.  A zero
// input gives +0 (never a negative-zero code).
__device__ __forceinline__ float expand_scaled(float x, float r, float k) {
    const float y = ex2_approx(fmaf(k, lg2_approx(r), kLog2_448));
    return __fadd_rn(copysignf(y, x), 0.0f);
}

// x / S ready for an E4M3 round-to-nearest-even conversion that rounds the
// EXACT quotient.  y = RN(x / S) can land exactly on a midpoint between two
// E4M3 values when the exact quotient lies just beside it; the exact remainder
// x - y S (an FMA, exact for a rounded quotient) tells which side, and y moves
// one float step that way.  No other midpoint can lie between y and the exact
// quotient (midpoints are floats, and the quotient is within half a float step
// of y), so this only matters when y is a midpoint.  Midpoints: 4 significant
// bits with the 4th set for |y| >= 2^-6, odd multiples of 2^-10 below.  S > 0.
// The remainder is exact only while it stays above the fp32 subnormal range:
// near a midpoint (>= 2^-10) of a quotient of an x below 2^-100 it can be
// about 2^-154 and round to zero, so such x and S are first scaled by 2^64
// (exact; the quotient is unchanged).
__device__ __forceinline__ float e4m3_quotient(float x, float S) {
    const float k = fabsf(x) < 0x1p-100f ? 0x1p64f : 1.0f;
    const float xs = x * k, Ss = S * k;
    const float y = __fdiv_rn(xs, Ss);
    const float ay = fabsf(y);
    const uint32_t b = __float_as_uint(ay);
    const float t = ay * 1024.0f;
    const bool mid = ay >= 0.015625f ? (b & 0xFFFFFu) == 0x80000u
                                     : (t == rintf(t) && (((uint32_t)t) & 1u) != 0u);
    const float r = fmaf(-y, Ss, xs);
    if (!mid || r == 0.0f) return y;
    return __uint_as_float(__float_as_uint(y) + (((r > 0.0f) == (y > 0.0f)) ? 1u : 0xFFFFFFFFu));
}

// E4M3 codes (round to nearest even, saturating, 0x00 for a zero) of the
// exact quotients x / S, S > 0, given inv ~ 1/S from the SFU (at most one
// float step off).  y = RN(x inv) is within 2.5 float steps of x / S;
// y (1 - 2^-20) and y (1 + 2^-20) lie at least 7.5 steps below and above it,
// so when both convert to the same code no E4M3 midpoint separates y from
// the exact quotient and that code is the answer.  The other elements (a
// midpoint within a few steps, or an SFU reciprocal that is not finite) are
// flagged in `undecided` and left to e4m3_code_of_quotient_exact.
constexpr float kDn = 0.99999904632568359f;   // 1 - 2^-20
constexpr float kUp = 1.00000095367431641f;   // 1 + 2^-20
__device__ __forceinline__ uint32_t e4m3_code_fast(float x, float inv, bool& undecided) {
    const float y = fmaf(x, inv, 0.0f);   // +0 for a zero of either sign
    const uint32_t p = e4m3x2(y * kDn, y * kUp);
    undecided = (p & 0xFFu) != (p >> 8) || !(inv <= 3.40282347e38f);
    return p & 0xFFu;
}
// The rare case, out of line so that it stays a branch taken by few lanes.
static __device__ __noinline__ uint32_t e4m3_code_of_quotient_exact(float x, float S) {
    return e4m3x2(__fadd_rn(e4m3_quotient(x, S), 0.0f), 0.0f) & 0xFFu;
}

// The exact codes of a pair of elements x0, x1 (scales S0, S1 > 0, normal)
// whose probe codes lo (of y (1 - 2^-20)) and hi (of y (1 + 2^-20)) may differ,
// 16 bits each.  The exact quotient x / S lies between the two probes, so its
// correctly rounded code is lo or hi, adjacent codes, and the midpoint
// between their values decides: the sign of 2|x| - (|lo| + |hi|) S, formed by
// one FMA (the sum is exact, and the FMA's rounding keeps the sign), says on
// which side the quotient lies; zero is a tie, which goes to the even code.
// A byte where lo and hi agree keeps its code.  The FMA could round a non-zero
// difference to zero only if it fell below 2^-149: its operands are multiples
// of 2^-142 or coarser unless |x| < 2^-100, and such an x (with S below 2^-89,
// as x / S is near a midpoint, at least 2^-11) is scaled with S by 2^64 first
// (exact).
__device__ __forceinline__ uint32_t e4m3x2_resolve(uint32_t lo, uint32_t hi, float x0, float x1, float S0,
                                                   float S1) {
    uint32_t hl, hh, hs;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(hl) : "h"((unsigned short)(lo & 0x7F7Fu)));
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(hh) : "h"((unsigned short)(hi & 0x7F7Fu)));
    asm("add.rn.f16x2 %0, %1, %2;" : "=r"(hs) : "r"(hl), "r"(hh));   // exact: 5 significant bits
    float s0, s1;
    asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.f32.f16 %0, a;\n\tcvt.f32.f16 %1, b;\n\t}"
        : "=f"(s0), "=f"(s1) : "r"(hs));
    const float a0 = fabsf(x0), a1 = fabsf(x1);
    const float k0 = a0 < 0x1p-100f ? 0x1p64f : 1.0f, k1 = a1 < 0x1p-100f ? 0x1p64f : 1.0f;
    float r0, r1;
    upk(fma2(pk(-s0, -s1), mul2(pk(S0, S1), pk(k0, k1)), mul2(pk(a0, a1), pk(2.0f * k0, 2.0f * k1))), r0, r1);
    const bool up0 = r0 > 0.0f || (r0 == 0.0f && (lo & 1u) != 0u);
    const bool up1 = r1 > 0.0f || (r1 == 0.0f && (lo & 0x100u) != 0u);
    return ((up0 ? hi : lo) & 0xFFu) | ((up1 ? hi : lo) & 0xFF00u);
}

// The stored code of a zero is 0x00 whatever the sign of the value that
// rounded to it: the conversion gives 0x80 for a negative value below half the
// smallest subnormal, and this clears the sign bit of every byte of a packed
// word whose low seven bits are all zero (bit 7 of (b & 0x7F) + 0x7F is set
// exactly when b & 0x7F is not zero; no byte carries into the next).
__device__ __forceinline__ uint32_t e4m3_canonical_zero(uint32_t w) {
    const uint32_t nz = (w & 0x7F7F7F7Fu) + 0x7F7F7F7Fu;
    return w & (nz | 0x7F7F7F7Fu);
}

// Smallest-non-zero tracking: fp32 magnitudes as unsigned bits minus one, so
// that zero wraps to 0xFFFFFFFF and never wins a min.
__device__ __forceinline__ uint32_t nz_key(float a) { return __float_as_uint(a) - 1u; }
__device__ __forceinline__ float nz_key_value(uint32_t key) { return __uint_as_float(key + 1u); }

}  // namespace coat
