// adamw_dre_step.cu -- the fused FP8 AdamW + Dynamic Range Expansion step for
// GB300 (sm_103a).
//
// One pass over HBM (COAT paper-review page, section 4 table, "fused optimizer
// kernel" row: the optimizer-state update is one fused CUDA kernel).  Per
// group of G contiguous parameters:
//   1. dequantize the E4M3 first/second moments and undo the expansion
//      (inverse of the section 3 FP8 quantization and f(x) = sign(x)|x|^k);
//   2. AdamW (section 3 core formulas): moment EMAs, bias correction,
//      decoupled weight decay, fp32 master weights from bf16 gradients;
//   3. two-stage max / smallest-non-zero reduction of |m_t| and v_t per group
//      (stage 1 per thread over 16 elements, stage 2 warp shuffles across the
//      G/16 lanes of the group);
//   4. fresh k = log_{R_X}(R_E4M3) and S = max^k / 448 per group and moment;
//   5. re-expand, round to E4M3 and store codes, weights and (S, k).
//
// Exact group extremes.  S = max^k / 448 with k = ln R_E4M3 / ln(max/min)
// amplifies a relative change of the group's max or min by up to ~30 (second
// moments: k ~ 4, log2 max ~ -25), and the smallest |m_t| of a group usually
// comes from a partial cancellation of beta1 m and (1 - beta1) g, where an
// fp32 evaluation has a large relative error.  So every element's moment is
// first computed on a fast fp32/SFU path whose error has a per-group bound;
// the elements whose fast value lies inside that bound around the group's
// fast max or min -- and the first moments so small that cancellation could
// move their code by more than one step -- are re-evaluated exactly:
// (|E4M3(q)| S)^(1/k) in double-float rounded once (a plain product when
// k = 1), then beta x + (1 - beta) g as a correctly rounded sum of two
// products.  The group's max and min are taken over those exact values, k and
// S are formed from them in double-float and rounded once, and the
// re-evaluated elements are encoded from their exact values.
//
// Execution.  A CTA of 128 threads owns 2048 consecutive parameters (16 per
// thread: every stream is whole 128-bit accesses); up to eight CTAs share an
// SM.  The per-group work runs as CTA-wide jobs between barriers -- one thread
// per (group, moment), and one to four threads per (group, statistic) -- so
// that it occupies a few full warps instead of a few lanes of every warp.  The
// moments wait in shared memory between phases; the exact pass reads a holder
// lane's gradients and codes again from L2.
//   B  stored-state parameters                      2 jobs per group
//   C  fast path, statistics, candidate holders      every thread
//   D  candidate masks and exact re-evaluation       4 jobs per group
//   E  k, S, encoding constants, record              2 jobs per group
//   F  encode and store codes                        every thread
// Groups of G < 16 parameters live inside one thread (step_kernel_thread).
#include <cstddef>

#include "coat_device.cuh"
#include <type_traits>

#include "coat_kernels.h"
#include "coat_round.cuh"

namespace coat {

// How often the exact path fell back to float64 because a double-float value
// lay too close to an fp32 rounding midpoint to round with certainty:
// [0] dequantized moments, [1] exponents k.  Only the rare path touches them.
__device__ unsigned long long g_recompute[2];

// The exact path reads its tables from their global copies (gtab), through
// L1: only the few lanes that re-evaluate candidates and the per-group jobs
// read them, so the step kernel's shared memory holds that path's inputs
// instead.
__device__ __forceinline__ df::Tables global_tables() {
    return df::Tables{reinterpret_cast<const df::LogEntry*>(gtab::kLog2Recip),
                      reinterpret_cast<const float*>(gtab::kExp2FracHi),
                      reinterpret_cast<const float*>(gtab::kExp2FracLo)};
}

namespace {

using df::F2;

constexpr unsigned kFull = 0xFFFFFFFFu;
#ifndef COAT_STEP_CTA
#define COAT_STEP_CTA 128
#endif
constexpr int kStepCta = COAT_STEP_CTA;    // threads per CTA of the step kernel
#define kInf __int_as_float(0x7F800000)

// Relative error bound of the SFU exp2 (ex2.approx.ftz.f32) for normal
// results; an exhaustive check over the arguments used here stays below it.
constexpr float kEx2Err = 2.384185791015625e-07f;   // 2^-22

// Bound on the relative error of a fast dequantized moment of a group whose
// stored exponent is k (1/k = rk): the SFU exp2 of the factor P and of the
// per-code term, the fp32 exponent log2(|E4M3(q)|/448) / k (|.| <= 17.81/k)
// rounded three times, and two roundings.
__device__ __forceinline__ float fast_err(float rk) {
    return 2.0f * kEx2Err + 1.5e-7f + 1.25e-07f * (17.81f * rk + 1.0f);
}

struct Chunk {
    float w[kVec];
    uint32_t g[kVec / 2];
    uint32_t mq[kVec / 4];
    uint32_t vq[kVec / 4];
};

__device__ __forceinline__ void load_chunk(const StepArgs& a, int64_t base, bool full, Chunk& c) {
    if (full) {
        const float4* wp = reinterpret_cast<const float4*>(a.w + base);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 v = ld_cs(wp + i);
            c.w[4 * i + 0] = v.x;
            c.w[4 * i + 1] = v.y;
            c.w[4 * i + 2] = v.z;
            c.w[4 * i + 3] = v.w;
        }
        // g and the codes keep the default cache policy (not evict-first): the
        // exact pass of this CTA reads some of them again a few microseconds later
        const uint4* gp = reinterpret_cast<const uint4*>(a.g + base);
        const uint4 g0 = __ldg(gp), g1 = __ldg(gp + 1);
        c.g[0] = g0.x; c.g[1] = g0.y; c.g[2] = g0.z; c.g[3] = g0.w;
        c.g[4] = g1.x; c.g[5] = g1.y; c.g[6] = g1.z; c.g[7] = g1.w;
        const uint4 m = __ldg(reinterpret_cast<const uint4*>(a.mq + base));
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(a.vq + base));
        c.mq[0] = m.x; c.mq[1] = m.y; c.mq[2] = m.z; c.mq[3] = m.w;
        c.vq[0] = v.x; c.vq[1] = v.y; c.vq[2] = v.z; c.vq[3] = v.w;
    } else {
#pragma unroll
        for (int i = 0; i < kVec / 2; ++i) c.g[i] = 0u;
#pragma unroll
        for (int i = 0; i < kVec / 4; ++i) { c.mq[i] = 0u; c.vq[i] = 0u; }
#pragma unroll
        for (int e = 0; e < kVec; ++e) {
            const bool in = base + e < a.n;
            c.w[e] = in ? a.w[base + e] : 0.0f;
            if (in) {
                c.g[e / 2] |= (uint32_t)a.g[base + e] << (16 * (e & 1));
                c.mq[e / 4] |= (uint32_t)a.mq[base + e] << (8 * (e & 3));
                c.vq[e / 4] |= (uint32_t)a.vq[base + e] << (8 * (e & 3));
            }
        }
    }
}

// The gradients and one moment's codes of the 16 parameters from `b`, read
// again from global memory (zero beyond n), as load_chunk packed them.
__device__ __forceinline__ void reload_inputs(const StepArgs& a, int64_t b, bool second, uint32_t* gw,
                                              uint32_t* cw) {
    const uint8_t* q = second ? a.vq : a.mq;
    if (b + kVec <= a.n) {
        const uint4* gp = reinterpret_cast<const uint4*>(a.g + b);
        const uint4 g0 = __ldg(gp), g1 = __ldg(gp + 1);
        const uint4 cc = __ldg(reinterpret_cast<const uint4*>(q + b));
        gw[0] = g0.x; gw[1] = g0.y; gw[2] = g0.z; gw[3] = g0.w;
        gw[4] = g1.x; gw[5] = g1.y; gw[6] = g1.z; gw[7] = g1.w;
        cw[0] = cc.x; cw[1] = cc.y; cw[2] = cc.z; cw[3] = cc.w;
    } else {
#pragma unroll
        for (int i = 0; i < kVec / 2; ++i) gw[i] = 0u;
#pragma unroll
        for (int i = 0; i < kVec / 4; ++i) cw[i] = 0u;
        for (int e = 0; e < kVec; ++e) {
            if (b + e < a.n) {
                gw[e / 2] |= (uint32_t)a.g[b + e] << (16 * (e & 1));
                cw[e / 4] |= (uint32_t)q[b + e] << (8 * (e & 3));
            }
        }
    }
}

// The same for both moments' codes at once.
__device__ __forceinline__ void reload_inputs_both(const StepArgs& a, int64_t b, uint32_t* gw, uint32_t* cm,
                                                   uint32_t* cv) {
    if (b + kVec <= a.n) {
        const uint4* gp = reinterpret_cast<const uint4*>(a.g + b);
        const uint4 g0 = __ldg(gp), g1 = __ldg(gp + 1);
        const uint4 m = __ldg(reinterpret_cast<const uint4*>(a.mq + b));
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(a.vq + b));
        gw[0] = g0.x; gw[1] = g0.y; gw[2] = g0.z; gw[3] = g0.w;
        gw[4] = g1.x; gw[5] = g1.y; gw[6] = g1.z; gw[7] = g1.w;
        cm[0] = m.x; cm[1] = m.y; cm[2] = m.z; cm[3] = m.w;
        cv[0] = v.x; cv[1] = v.y; cv[2] = v.z; cv[3] = v.w;
    } else {
        reload_inputs(a, b, false, gw, cm);
        reload_inputs(a, b, true, gw, cv);
    }
}

// Bulk prefetch of `bytes` (a multiple of 16) at a 16-byte aligned address into
// L2 (cp.async.bulk.prefetch: no registers, no shared memory, no completion
// to wait for).
__device__ __forceinline__ void l2_prefetch(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}
constexpr int kL2Ahead = 608;   // CTAs between a CTA and the tile it prefetches

__device__ __forceinline__ void zero_chunk(Chunk& c) {
#pragma unroll
    for (int e = 0; e < kVec; ++e) c.w[e] = 0.0f;
#pragma unroll
    for (int i = 0; i < kVec / 2; ++i) c.g[i] = 0u;
#pragma unroll
    for (int i = 0; i < kVec / 4; ++i) { c.mq[i] = 0u; c.vq[i] = 0u; }
}

__device__ __forceinline__ void store_w(const StepArgs& a, int64_t base, bool full, const Chunk& c) {
    if (full) {
        float4* wp = reinterpret_cast<float4*>(a.w + base);
#pragma unroll
        for (int i = 0; i < 4; ++i)
            st_cs(wp + i, make_float4(c.w[4 * i], c.w[4 * i + 1], c.w[4 * i + 2], c.w[4 * i + 3]));
    } else {
#pragma unroll
        for (int e = 0; e < kVec; ++e)
            if (base + e < a.n) a.w[base + e] = c.w[e];
    }
}

__device__ __forceinline__ uint32_t byte_of(const uint32_t* w, int j) {
    return (w[j >> 2] >> (8 * (j & 3))) & 0xFFu;
}
__device__ __forceinline__ float bf16_of(const uint32_t* w, int j) {
    return (j & 1) ? __uint_as_float(w[j >> 1] & 0xFFFF0000u) : __uint_as_float(w[j >> 1] << 16);
}

// Value of a non-negative E4M3 magnitude code (bias 7, subnormal below 8).
__device__ __forceinline__ float e4m3_value(uint32_t mag) {
    return mag >= 8u ? __uint_as_float((((mag >> 3) + 120u) << 23) | ((mag & 7u) << 20))
                     : __fmul_rn((float)mag, 0.001953125f);
}

// Parameters of one stored moment.  Exact path: A = log2(448 S) and 1/k as
// double-floats (and S itself for k = 1).  Fast path: P = (448 S)^(1/k), 1/k.
struct StateParams {
    F2 A;
    F2 rkd;
    float P;
    float S;
};

__device__ __forceinline__ StateParams state_params(float S, float k, const df::Tables& t) {
    StateParams p;
    p.S = S;
    p.rkd = df::recip21(k);
    if (S > 0.0f) {
        p.A = df::add2(df::log2_df(S, t), const_df(kLog2_448Df));
        const F2 z = df::mul22(p.A, p.rkd);                 // log2 P
        const float n = rintf(z.hi);
        p.P = df::scale2(ex2_ftz(__fadd_rn(__fsub_rn(z.hi, n), z.lo)), (int)n);
    } else {
        p.A = F2{-1e30f, 0.0f};
        p.P = 0.0f;
    }
    return p;
}

// Exactly rounded new moment of one element:
//   prev = sign(q) RN((|E4M3(q)| S)^(1/k)),  RN(beta prev + (1-beta) x),
// with x = g (first moment) or g^2 (second moment, exact for a bf16 g).
// For k = 1 the power is the plain product |E4M3(q)| S, which is often a
// rounding tie: it is formed by one correctly rounded multiplication.
// Otherwise the power is rounded with certainty (float64 in the rare case
// where the double-float value lies too near an fp32 rounding midpoint; only
// that case calls k_of() for the stored exponent).
template <typename KOf>
__device__ __forceinline__ float exact_moment(uint32_t code, float gf, bool second, F2 A, F2 rkd,
                                              float S, KOf k_of, float beta, float omb,
                                              const df::Tables& t, const float* lg_hi,
                                              const float* lg_lo) {
    float prev = 0.0f;
    const uint32_t mag = code & 0x7Fu;
    if (mag != 0u && S > 0.0f) {
        if (rkd.hi == 1.0f && rkd.lo == 0.0f) {
            prev = __fmul_rn(e4m3_value(mag), S);
        } else {
            const F2 L = {lg_hi[mag], lg_lo[mag]};
            bool slow = false;
            prev = df::dequant_try(L, A, rkd, t, slow);
            if (slow) {
                prev = df::dequant_f64(e4m3_value(mag), S, k_of());
                atomicAdd(&g_recompute[0], 1ull);
            }
        }
        if (code & 0x80u) prev = -prev;
    }
    const float x = second ? __fmul_rn(gf, gf) : gf;
    return df::dot2_rn(beta, prev, omb, x);
}

// k correctly rounded from double-float logs of the group's max / min
// magnitudes (Lmx, Lmn: log2 of mx, mn), with the cap and the S-range guard;
// S = 2^(k log2 max - log2 448) rounded once.
__device__ __forceinline__ void k_and_S_logs(float mx, float mn, F2 Lmx, F2 Lmn,
                                             const df::Tables& t, float& k, float& S) {
    if (!(mx > 0.0f)) {
        k = 1.0f;
        S = 0.0f;
        return;
    }
    bool slow = false;
    k = df::k_certain(mx, mn, Lmx, Lmn, k_consts(), slow);
    if (slow) atomicAdd(&g_recompute[1], 1ull);
    S = df::exp2_df(df::add2(df::mul21(Lmx, k), df::neg2(const_df(kLog2_448Df))), t);
}

// The same with the logs formed here.
__device__ __forceinline__ void k_and_S(float mx, float mn, const df::Tables& t, float& k,
                                        float& S) {
    if (!(mx > 0.0f)) {
        k = 1.0f;
        S = 0.0f;
        return;
    }
    const F2 Lmx = df::log2_df(mx, t);
    const F2 Lmn = (mn > 0.0f && mn < mx) ? df::log2_df(mn, t) : Lmx;
    k_and_S_logs(mx, mn, Lmx, Lmn, t, k, S);
}

// Encoding constants: r = |x| * inv, y = 2^(k log2 r + cz).  A subnormal max
// is pre-scaled by 2^24 (inv = 1/(max 2^24)) and the factor folded into cz.
__device__ __forceinline__ void encode_consts(float mx, float k, float& inv, float& cz) {
    const bool sub = mx < 1.17549435e-38f;
    inv = mx > 0.0f ? __frcp_rn(sub ? mx * 16777216.0f : mx) : 0.0f;
    cz = sub ? fmaf(24.0f, k, kLog2_448) : kLog2_448;
}

// Three-input minimum / maximum (PTX min/max with three operands, sm_100 and
// later).  A NaN operand is ignored unless every operand is NaN.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
__device__ __forceinline__ float fmin3(float a, float b, float c) {
    float d;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Smallest-non-zero keys: |bits(x) - 1| read as a float orders like |x| for
// x != 0 and is NaN for +-0, which min ignores.  A minimum of keys started at
// +inf stays +inf when every value is zero.
__device__ __forceinline__ float nz_key(float x) {
    return fabsf(__uint_as_float(__float_as_uint(x) - 1u));
}
__device__ __forceinline__ float nz_key_value(float k) {
    return k < kInf ? __uint_as_float(__float_as_uint(k) + 1u) : 0.0f;
}

// Byte offset of the table entry of code byte i of a packed word (magnitude
// bits only): ((w >> 8i) & 0x7F) * 4 with one shift and one mask.
template <int I>
__device__ __forceinline__ uint32_t code_off(uint32_t w) {
    if constexpr (I == 0) return (w << 2) & 0x1FCu;
    else return (w >> (8 * I - 2)) & 0x1FCu;
}
__device__ __forceinline__ float table_at(const float* t, uint32_t off) {
    return *reinterpret_cast<const float*>(reinterpret_cast<const char*>(t) + off);
}

// Fast path of one element: dequantize, EMAs, AdamW.  bPm = beta1 P_m and
// bPv = beta2 P_v per group; the first moment's code sign flips bPm, and
// (1 - beta1) g is formed as fma(.., .., +0) so that m_t is never -0.  SFU
// ops flush below 2^-126 only.
template <int I>
__device__ __forceinline__ void fast_elem(const StepArgs& a, uint32_t wm, uint32_t wv, float gf,
                                          float& w, const float* lg, float bPm, float rkm,
                                          float bPv, float rkv, float& mt, float& vt) {
    const float em = ex2_ftz(__fmul_rn(table_at(lg, code_off<I>(wm)), rkm));
    const float ev = ex2_ftz(__fmul_rn(table_at(lg, code_off<I>(wv)), rkv));
    const float bPs = __uint_as_float(__float_as_uint(bPm) ^ ((wm << (24 - 8 * I)) & 0x80000000u));
    mt = fmaf(bPs, em, fmaf(a.omb1, gf, 0.0f));
    vt = fmaf(bPv, ev, __fmul_rn(__fmul_rn(a.omb2, gf), gf));
    // -c1 / (sqrt(v c2) + eps) as 1 / (sqrt(v) sq + ep); sqrt.approx of a v below
    // 2^-126 is 0, where eps dominates the denominator
    w = fmaf(mt, rcp_ftz(fmaf(sqrt_ftz(vt), a.sq, a.ep)), __fmul_rn(w, a.decay));
}

// Elements I and I + 1 of a packed word on the packed f32x2 path: every
// product and FMA is the scalar one of fast_elem, two lanes per instruction.
template <int I>
__device__ __forceinline__ void fast_pair(const StepArgs& a, uint32_t wm, uint32_t wv, float g0, float g1,
                                          float& w0, float& w1, const float* lg, float bPm, float rkm,
                                          float bPv, float rkv, float& m0, float& m1, float& v0, float& v1) {
    float pm0, pm1, pv0, pv1;
    upk(mul2(pk(table_at(lg, code_off<I>(wm)), table_at(lg, code_off<I + 1>(wm))), pk(rkm, rkm)), pm0, pm1);
    upk(mul2(pk(table_at(lg, code_off<I>(wv)), table_at(lg, code_off<I + 1>(wv))), pk(rkv, rkv)), pv0, pv1);
    const float bPs0 = __uint_as_float(__float_as_uint(bPm) ^ ((wm << (24 - 8 * I)) & 0x80000000u));
    const float bPs1 = __uint_as_float(__float_as_uint(bPm) ^ ((wm << (16 - 8 * I)) & 0x80000000u));
    const uint64_t gg = pk(g0, g1);
    const uint64_t mt = fma2(pk(bPs0, bPs1), pk(ex2_ftz(pm0), ex2_ftz(pm1)), fma2(pk(a.omb1, a.omb1), gg, pk(0.0f, 0.0f)));
    const uint64_t vt = fma2(pk(bPv, bPv), pk(ex2_ftz(pv0), ex2_ftz(pv1)), mul2(mul2(pk(a.omb2, a.omb2), gg), gg));
    upk(mt, m0, m1);
    upk(vt, v0, v1);
    float d0, d1;
    upk(fma2(pk(sqrt_ftz(v0), sqrt_ftz(v1)), pk(a.sq, a.sq), pk(a.ep, a.ep)), d0, d1);
    upk(fma2(mt, pk(rcp_ftz(d0), rcp_ftz(d1)), mul2(pk(w0, w1), pk(a.decay, a.decay))), w0, w1);
}

__device__ __forceinline__ uint32_t encode_pair_m(float m0, float m1, float k, float inv, float cz) {
    float a0, a1, b0, b1;
    upk(mul2(pk(fabsf(m0), fabsf(m1)), pk(inv, inv)), a0, a1);
    upk(fma2(pk(k, k), pk(lg2_ftz(a0), lg2_ftz(a1)), pk(cz, cz)), b0, b1);
    return e4m3x2(copysignf(ex2_ftz(b0), m0), copysignf(ex2_ftz(b1), m1));
}
__device__ __forceinline__ uint32_t encode_pair_v(float v0, float v1, float k, float inv, float cz) {
    float a0, a1, b0, b1;
    upk(mul2(pk(v0, v1), pk(inv, inv)), a0, a1);
    upk(fma2(pk(k, k), pk(lg2_ftz(a0), lg2_ftz(a1)), pk(cz, cz)), b0, b1);
    return e4m3x2(ex2_ftz(b0), ex2_ftz(b1));
}

// ---------------------------------------------------------------------------
// G >= 16: CTA-cooperative kernel
// ---------------------------------------------------------------------------

// Candidate windows of one group, built from its fast statistics.  With
// T_j = |beta1 m_prev,j| + (1 - beta1)|g_j| <= |m_j| + 2 (1 - beta1)|g_j| and
// T the same bound over the group, a fast m_j is within eps_m T_j of its
// exact value and a fast v_j within eps_v v_j, so:
//   max|m|:  the true max has |m_j| >= fmx_m - 2 eps_m T;
//   min|m|:  the true smallest non-zero has |m_j| <= fmn_m + eps_m (T_j + T);
//            and every |m_j| <= 2^10 eps_m T_j (relative error above 2^-10,
//            where cancellation could move the code by more than one step)
//            is re-evaluated too;
//   max v:   v_j >= fmx_v (1 - 2 eps_v);   min v: v_j <= fmn_v (1 + 4 eps_v).
struct GroupWin {
    float hi_m, fmn_m, eps_m, T, hi_v, lo_v;
};

__device__ __forceinline__ GroupWin make_win(const StepArgs& a, float P_m, float eps_m, float eps_v,
                                             float fmx_m, float fmn_m, float fmx_v, float fmn_v,
                                             float gmx) {
    GroupWin w;
    w.T = fmaf(a.beta1, P_m * (1.0f + eps_m), a.omb1 * gmx);
    w.eps_m = eps_m;
    w.hi_m = fmx_m - 2.0f * eps_m * w.T;
    w.fmn_m = fmn_m;
    w.hi_v = fmx_v * (1.0f - 2.0f * eps_v);
    w.lo_v = fmn_v > 0.0f ? fmn_v * (1.0f + 4.0f * eps_v) : -1.0f;
    return w;
}

// Candidate test of statistic s as one branch-free expression (a job's lanes
// run different statistics): max statistics test |x| >= hi; min statistics
// test |x| <= max(a0 + a1 T_j, a2 T_j) with T_j = |x| + c |g| (c = 2(1-beta1)
// for m, 0 for v).
struct CandTest {
    bool is_max;
    float hi, a0, a1, a2, c;
};

__device__ __forceinline__ CandTest cand_test(const GroupWin& w, int s, float omb1) {
    CandTest t;
    t.is_max = (s & 1) == 0;
    t.hi = (s == 0) ? w.hi_m : w.hi_v;
    const bool m_min = (s == 1);
    t.a0 = m_min ? (w.fmn_m > 0.0f ? fmaf(w.eps_m, w.T, w.fmn_m) : -kInf) : w.lo_v;
    t.a1 = m_min ? w.eps_m : 0.0f;
    t.a2 = m_min ? 1024.0f * w.eps_m : 0.0f;
    t.c = m_min ? 2.0f * omb1 : 0.0f;
    return t;
}

// `code` is the element's stored code byte.  A fast value of exactly zero is
// tested too unless the element's inputs are both zero (g = 0 and a zero
// code, whose moment is exactly 0): the fast sum can cancel to 0 where the
// exact one does not, and an SFU flush can zero a tiny non-zero term.
__device__ __forceinline__ bool cand(float x, float gabs, uint32_t code, const CandTest& t) {
    const float ax = fabsf(x);
    const float Tj = fmaf(t.c, gabs, ax);
    const float lo = fmaxf(fmaf(t.a1, Tj, t.a0), t.a2 * Tj);
    const bool live = ax > 0.0f || gabs > 0.0f || (code & 0x7Fu) != 0u;
    return live && (t.is_max ? ax >= t.hi : ax <= lo);
}

// Per-group shared-memory record (index of the group within the CTA).
struct GroupRec {
    F2 A[2];             // log2(448 S) of the stored m (0) and v (1)
    F2 rkd[2];           // 1/k
    F2 lex[4];           // log2 of the exact extremes
    float P[2];          // fast-path factor
    float S[2];          // stored S
    float fmx[2];        // fast max |m|, max v
    float fmn[2];        // fast smallest non-zero
    float gmx;           // max |g|
    uint32_t hwarp;      // warp holding the group
    uint32_t holders[4]; // lanes holding candidates, per statistic
    float ex[4];         // exact extremes
    float k[2];          // fresh k
    float inv[2];        // encoding constants
    float cz[2];
};

// The records of a CTA's N groups in shared memory, either as an array of
// GroupRec or (kSoA) as a structure of arrays.  The per-group jobs of G <= 32
// run one group per lane (statistic blocks): lanes then read one field of
// consecutive groups, which the structure of arrays puts in consecutive words;
// for larger G the four jobs of a group sit on adjacent lanes and read
// neighbouring fields of one record.
template <int N, bool kSoA>
struct GroupRecs {
    unsigned char* p;
#define COAT_REC_FIELD(T, name, M)                                                                   \
    __device__ __forceinline__ T& name(int m, int i) const {                                        \
        if constexpr (kSoA)                                                                          \
            return reinterpret_cast<T*>(p + (size_t)N * offsetof(GroupRec, name))[m * N + i];         \
        else                                                                                         \
            return reinterpret_cast<GroupRec*>(p)[i].name[m];                                        \
    }
    COAT_REC_FIELD(F2, A, 2)
    COAT_REC_FIELD(F2, rkd, 2)
    COAT_REC_FIELD(F2, lex, 4)
    COAT_REC_FIELD(float, P, 2)
    COAT_REC_FIELD(float, S, 2)
    COAT_REC_FIELD(float, fmx, 2)
    COAT_REC_FIELD(float, fmn, 2)
    COAT_REC_FIELD(uint32_t, holders, 4)
    COAT_REC_FIELD(float, ex, 4)
    COAT_REC_FIELD(float, k, 2)
    COAT_REC_FIELD(float, inv, 2)
    COAT_REC_FIELD(float, cz, 2)
#undef COAT_REC_FIELD
    __device__ __forceinline__ float& gmx(int i) const {
        if constexpr (kSoA) return reinterpret_cast<float*>(p + (size_t)N * offsetof(GroupRec, gmx))[i];
        else return reinterpret_cast<GroupRec*>(p)[i].gmx;
    }
    __device__ __forceinline__ uint32_t& hwarp(int i) const {
        if constexpr (kSoA) return reinterpret_cast<uint32_t*>(p + (size_t)N * offsetof(GroupRec, hwarp))[i];
        else return reinterpret_cast<GroupRec*>(p)[i].hwarp;
    }
};

// Moment rows: 16 floats per thread, the four 16-byte chunks of thread t
// stored in the order q ^ ((t >> 1) & 3): 128-bit accesses by consecutive
// threads hit distinct bank groups.
__device__ __forceinline__ int chunk_slot(int t, int q) { return 4 * (q ^ ((t >> 1) & 3)); }

template <int G, int CTA>
struct CtaLayout {
    static constexpr int kCtaElems = CTA * kVec;  // parameters per CTA
    static constexpr int NGC = kCtaElems / G;   // groups per CTA
    static constexpr int L = G / kVec;          // lanes per group
    static constexpr size_t off_m = 0;
    static constexpr size_t off_v = off_m + (size_t)CTA * kVec * 4;
    static constexpr size_t off_grp = off_v + (size_t)CTA * kVec * 4;
    static constexpr size_t off_lg = off_grp + (size_t)NGC * sizeof(GroupRec);
    static constexpr size_t bytes = off_lg + 128 * 4;
};

template <int G, int CTA>
__global__ void __launch_bounds__(CTA, 1024 / CTA)   // 64 registers: 1024 threads per SM
step_kernel_cta(const StepArgs a) {
    using Lay = CtaLayout<G, CTA>;
    constexpr int kCta = CTA;
    constexpr int kCtaElems = Lay::kCtaElems;
    constexpr int NGC = Lay::NGC;
    constexpr int L = Lay::L;
    static_assert(L >= 1 && L <= 16 && (Lay::off_v % 16) == 0 && (Lay::off_grp % 16) == 0 &&
                      (Lay::off_lg % 4) == 0,
                  "shared-memory layout");
    extern __shared__ __align__(16) unsigned char smem[];
    float(*sm_m)[kVec] = reinterpret_cast<float(*)[kVec]>(smem + Lay::off_m);
    float(*sm_v)[kVec] = reinterpret_cast<float(*)[kVec]>(smem + Lay::off_v);
    const GroupRecs<NGC, (NGC >= 64)> R{smem + Lay::off_grp};   // structure of arrays with statistic blocks
    float* lg_hi = reinterpret_cast<float*>(smem + Lay::off_lg);
    const float* lg_lo = reinterpret_cast<const float*>(gtab::kLog2Frac448Lo);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t cta_base = (int64_t)blockIdx.x * kCtaElems;
    const int64_t g_first = cta_base / G;
    const int64_t base = cta_base + (int64_t)tid * kVec;
    const bool active = base < a.n;
    const bool full = base + kVec <= a.n;

    // Bulk L2 prefetch of the tile of the CTA kL2Ahead launches later (roughly
    // half a wave on GB300): its DRAM reads start while this CTA computes, so
    // more requests are in flight than the CTAs' own loads keep (3.7 % off the
    // Llama-2-7B step).  One thread, four bulk prefetches, and for G <= 32 a
    // fifth for the group records (phase B reads them first and every warp
    // waits for B: 2.7 % off the step at G = 16 and 32; no gain at G = 64, and
    // at G = 128 the 256 bytes are not worth the extra request); a tile that
    // ends past n is not prefetched.
    {
        const int64_t pf = cta_base + (int64_t)kL2Ahead * kCtaElems;
        if (tid == 0 && pf + kCtaElems <= a.n) {
            if constexpr (G <= 32) l2_prefetch(a.meta + pf / G, NGC * 16);
            l2_prefetch(a.w + pf, kCtaElems * 4);
            l2_prefetch(a.g + pf, kCtaElems * 2);
            l2_prefetch(a.mq + pf, kCtaElems);
            l2_prefetch(a.vq + pf, kCtaElems);
        }
    }
    // the stored records of B's jobs first, then this thread's parameters: the
    // loads are in flight during phase B
    float2 bsk[(2 * NGC + kCta - 1) / kCta];
#pragma unroll
    for (int i = 0; i < (2 * NGC + kCta - 1) / kCta; ++i) {
        const int j = tid + i * kCta;
        bsk[i] = make_float2(0.0f, 1.0f);
        const int64_t gg = g_first + (j >> 1);
        if (j < 2 * NGC && gg * G < a.n) bsk[i] = reinterpret_cast<const float2*>(a.meta + gg)[j & 1];
    }
    Chunk c;
    if (active) load_chunk(a, base, full, c);
    else zero_chunk(c);

    for (int i = tid; i < 128; i += kCta) lg_hi[i] = __uint_as_float(gtab::kLog2Frac448Hi[i]);
    __syncthreads();
    const df::Tables tab = global_tables();

    // ---- B: stored-state parameters, one job per (group, moment) ----
#pragma unroll
    for (int i = 0; i < (2 * NGC + kCta - 1) / kCta; ++i) {
        const int j = tid + i * kCta;
        if (j >= 2 * NGC) break;
        const int gi = j >> 1, sm_ = j & 1;
        const float S = bsk[i].x, k = bsk[i].y;
        const StateParams p = state_params(S, k, tab);
        const int ri = gi;
        R.A(sm_, ri) = p.A;
        R.rkd(sm_, ri) = p.rkd;
        R.P(sm_, ri) = p.P;
        R.S(sm_, ri) = S;
    }
    __syncthreads();

    // ---- C: fast path, statistics, candidate holders ----
    const int gi = (tid * kVec) / G;
    const int lig = (tid * kVec % G) / kVec;   // lane within the group
    {
        const int ri = gi;
        const float Pm = R.P(0, ri), rkm = R.rkd(0, ri).hi, rkv = R.rkd(1, ri).hi;
        const float bPm = a.beta1 * Pm, bPv = a.beta2 * R.P(1, ri);
        float lmx_m = 0.0f, lmx_v = 0.0f, lmx_g = 0.0f;
        float lmn_m = kInf, lmn_v = kInf;   // smallest |m| and v, zeros included
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float mt[4], vt[4];
            const float g0 = bf16_of(c.g, 4 * q), g1 = bf16_of(c.g, 4 * q + 1);
            const float g2 = bf16_of(c.g, 4 * q + 2), g3 = bf16_of(c.g, 4 * q + 3);
            fast_pair<0>(a, c.mq[q], c.vq[q], g0, g1, c.w[4 * q], c.w[4 * q + 1], lg_hi, bPm, rkm, bPv, rkv,
                         mt[0], mt[1], vt[0], vt[1]);
            fast_pair<2>(a, c.mq[q], c.vq[q], g2, g3, c.w[4 * q + 2], c.w[4 * q + 3], lg_hi, bPm, rkm, bPv,
                         rkv, mt[2], mt[3], vt[2], vt[3]);
            lmx_g = fmax3(fmax3(lmx_g, fabsf(g0), fabsf(g1)), fabsf(g2), fabsf(g3));
            lmx_m = fmax3(fmax3(lmx_m, fabsf(mt[0]), fabsf(mt[1])), fabsf(mt[2]), fabsf(mt[3]));
            lmx_v = fmax3(fmax3(lmx_v, vt[0], vt[1]), vt[2], vt[3]);
            lmn_m = fmin3(fmin3(lmn_m, fabsf(mt[0]), fabsf(mt[1])), fabsf(mt[2]), fabsf(mt[3]));
            lmn_v = fmin3(fmin3(lmn_v, vt[0], vt[1]), vt[2], vt[3]);
            const int slot = chunk_slot(tid, q);
            *reinterpret_cast<float4*>(&sm_m[tid][slot]) = make_float4(mt[0], mt[1], mt[2], mt[3]);
            *reinterpret_cast<float4*>(&sm_v[tid][slot]) = make_float4(vt[0], vt[1], vt[2], vt[3]);
        }
        if (active) store_w(a, base, full, c);

        // smallest non-zero values as keys; a lane holding an exact zero (rare:
        // both inputs of an element zero, or a fast sum that cancels) rescans
        // its values
        const float lz = fminf(lmn_m, lmn_v);   // zero iff a fast value is zero
        lmn_m = nz_key(lmn_m);
        lmn_v = nz_key(lmn_v);
        if (lz == 0.0f) {
            lmn_m = kInf;
            lmn_v = kInf;
#pragma unroll 1
            for (int e = 0; e < kVec; ++e) {
                lmn_m = fminf(lmn_m, nz_key(sm_m[tid][e]));
                lmn_v = fminf(lmn_v, nz_key(sm_v[tid][e]));
            }
        }

        // stage 2 across the lanes of the group
        float fmx_m = lmx_m, fmx_v = lmx_v, gmx = lmx_g, fmn_m = lmn_m, fmn_v = lmn_v;
#pragma unroll
        for (int off = L / 2; off > 0; off >>= 1) {
            fmx_m = fmaxf(fmx_m, __shfl_xor_sync(kFull, fmx_m, off));
            fmx_v = fmaxf(fmx_v, __shfl_xor_sync(kFull, fmx_v, off));
            gmx = fmaxf(gmx, __shfl_xor_sync(kFull, gmx, off));
            fmn_m = fminf(fmn_m, __shfl_xor_sync(kFull, fmn_m, off));
            fmn_v = fminf(fmn_v, __shfl_xor_sync(kFull, fmn_v, off));
        }
        const float fmn_mv = nz_key_value(fmn_m), fmn_vv = nz_key_value(fmn_v);
        const GroupWin win = make_win(a, Pm, fast_err(rkm), fast_err(rkv), fmx_m, fmn_mv, fmx_v, fmn_vv, gmx);
        // lane-level tests: sufficient conditions for holding a candidate.  A
        // lane with a fast zero holds one when the group has a non-zero input.
        const bool live_m = win.T > 0.0f, live_v = R.P(1, ri) > 0.0f || gmx > 0.0f;
        const float lmn_mv = nz_key_value(lmn_m), lmn_vv = nz_key_value(lmn_v);
        const float Tl = fmaf(2.0f * a.omb1, lmx_g, lmx_m);   // >= T_j of every element here
        const bool c1 = (lmn_mv > 0.0f &&
                         ((fmn_mv > 0.0f && lmn_mv <= fmaf(win.eps_m, Tl + win.T, fmn_mv)) ||
                          lmn_mv <= 1024.0f * win.eps_m * Tl)) ||
                        (lz == 0.0f && live_m);
        const uint32_t gmask = ((1u << L) - 1u) << (lane - lig);
        const uint32_t h0 = __ballot_sync(kFull, lmx_m >= win.hi_m && (lmx_m > 0.0f || live_m)) & gmask;
        const uint32_t h1 = __ballot_sync(kFull, c1) & gmask;
        const uint32_t h2 = __ballot_sync(kFull, lmx_v >= win.hi_v && (lmx_v > 0.0f || live_v)) & gmask;
        const uint32_t h3 = __ballot_sync(kFull, (lmn_vv > 0.0f && lmn_vv <= win.lo_v) ||
                                                     (lz == 0.0f && live_v)) & gmask;
        if (lig == 0) {
            R.fmx(0, ri) = fmx_m;
            R.fmx(1, ri) = fmx_v;
            R.fmn(0, ri) = fmn_mv;
            R.fmn(1, ri) = fmn_vv;
            R.gmx(ri) = gmx;
            R.hwarp(ri) = (uint32_t)warp;
            R.holders(0, ri) = h0;
            R.holders(1, ri) = h1;
            R.holders(2, ri) = h2;
            R.holders(3, ri) = h3;
        }
    }
    __syncthreads();

    // ---- D: candidates re-evaluated exactly, one job per (group, statistic) ----
    // A job may read a value another job of the same group has already
    // replaced by its exact value; the windows hold the exact values of the
    // true extremes too, so the outcome is the same.
    // With 64 or more groups per CTA (G <= 32) the jobs run in blocks of NGC per
    // statistic (max m, max v, min m, min v), so every job warp of a pass runs
    // one kind of window test and the passes are balanced; with fewer groups a
    // block would leave the minimum jobs to a single warp, and the jobs of a
    // group stay on adjacent lanes instead.
    constexpr bool kStatBlocks = NGC >= 64;
    // With G >= 128 the 4 NGC jobs would leave half or more of the CTA idle:
    // a group gets kT = 128 / NGC threads instead (8 or 16).  Its lanes 0, 1, 2
    // take max|m|, max v and min v, whose windows admit one holder lane almost
    // always; the other kT - 3 share the holder lanes of min|m| (partial
    // cancellation puts two or three lanes in its window), scanning every
    // (kT - 3)-th of them, and combine their minima by shuffles over the kT lanes.
    constexpr int kT = (kCta % NGC == 0) ? kCta / NGC : 0;
    constexpr bool kAsym = kT >= 8 && L >= 4;
    static_assert(!kAsym || (32 % kT == 0 && kT * NGC == kCta), "a group's lanes within one warp");
    constexpr bool kOwnGroup = kStatBlocks && L == 1 && kCta == NGC;
    if constexpr (kOwnGroup) {
        // G = 16: a thread holds one whole group and runs its four statistics
        // itself: the windows formed once, its inputs read again once, each
        // statistic's test specialised, and the four logs side by side.
        const int ri = tid;
        const GroupWin win = make_win(a, R.P(0, ri), fast_err(R.rkd(0, ri).hi), fast_err(R.rkd(1, ri).hi),
                                      R.fmx(0, ri), R.fmn(0, ri), R.fmx(1, ri), R.fmn(1, ri), R.gmx(ri));
        const uint32_t hol[4] = {R.holders(0, ri), R.holders(1, ri), R.holders(2, ri), R.holders(3, ri)};
        uint32_t gw[8], cm[4], cv[4];
#pragma unroll
        for (int i = 0; i < 8; ++i) gw[i] = 0u;
#pragma unroll
        for (int i = 0; i < 4; ++i) { cm[i] = 0u; cv[i] = 0u; }
        if ((hol[0] | hol[1] | hol[2] | hol[3]) != 0u) reload_inputs_both(a, base, gw, cm, cv);
        float best[4];
        const auto one = [&](auto sc) {
            constexpr int St = decltype(sc)::value;
            constexpr bool second = St >= 2, is_max = (St & 1) == 0;
            constexpr int sm_ = second ? 1 : 0;
            float bst = is_max ? 0.0f : kInf;
            if (hol[St] != 0u) {
                const CandTest ct = cand_test(win, St, a.omb1);
                const F2 A = R.A(sm_, ri), rkd = R.rkd(sm_, ri);
                const float S = R.S(sm_, ri);
                const float* kst_at = reinterpret_cast<const float*>(a.meta + g_first + ri) + 2 * sm_ + 1;
                const auto kst = [kst_at]() { return *kst_at; };
                const float beta = second ? a.beta2 : a.beta1, omb = second ? a.omb2 : a.omb1;
                float* vals = second ? sm_v[tid] : sm_m[tid];
                const uint32_t* cw = second ? cv : cm;
                uint32_t msk = 0u, zm = 0u;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 x4 = *reinterpret_cast<const float4*>(vals + chunk_slot(tid, q));
                    const float xs[4] = {x4.x, x4.y, x4.z, x4.w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float ax = fabsf(xs[i]);
                        bool in;
                        if constexpr (is_max) {
                            in = ax >= ct.hi;
                        } else if constexpr (second) {
                            in = ax <= fmaxf(ct.a0, 0.0f);
                        } else {
                            const float Tj = fmaf(ct.c, fabsf(bf16_of(gw, 4 * q + i)), ax);
                            in = ax <= fmaxf(fmaf(ct.a1, Tj, ct.a0), ct.a2 * Tj);
                        }
                        msk |= (in ? 1u : 0u) << (4 * q + i);
                        zm |= (ax == 0.0f ? 1u : 0u) << (4 * q + i);
                    }
                }
                // a max window admits zeros only when degenerate; a zero is a
                // candidate only when its inputs are not both zero
                if constexpr (is_max) {
                    if (ct.hi > 0.0f) zm = 0u;
                }
                uint32_t zc = msk & zm;
                while (zc) {
                    const int e = __ffs(zc) - 1;
                    zc &= zc - 1u;
                    if (bf16_of(gw, e) == 0.0f && (byte_of(cw, e) & 0x7Fu) == 0u) msk &= ~(1u << e);
                }
                while (msk) {
                    const int e = __ffs(msk) - 1;
                    msk &= msk - 1u;
                    const float x = exact_moment(byte_of(cw, e), bf16_of(gw, e), second, A, rkd, S, kst, beta,
                                                 omb, tab, lg_hi, lg_lo);
                    vals[chunk_slot(tid, e >> 2) + (e & 3)] = x;   // encoded from the exact value
                    const float ax = fabsf(x);
                    if (is_max) bst = fmaxf(bst, ax);
                    else if (ax > 0.0f) bst = fminf(bst, ax);
                }
            }
            best[St] = (bst < kInf) ? bst : 0.0f;
        };
        one(std::integral_constant<int, 0>{});
        one(std::integral_constant<int, 2>{});
        one(std::integral_constant<int, 1>{});
        one(std::integral_constant<int, 3>{});
        F2 lx[4];
#pragma unroll
        for (int st = 0; st < 4; ++st) lx[st] = best[st] > 0.0f ? df::log2_df(best[st], tab) : F2{0.0f, 0.0f};
#pragma unroll
        for (int st = 0; st < 4; ++st) {
            R.ex(st, ri) = best[st];
            R.lex(st, ri) = lx[st];
        }
    }
    for (int jt = tid; jt < (kOwnGroup ? 0 : (kAsym ? kCta : 4 * NGC)); jt += kCta) {
        const int j = jt;
        int jg, s, sub = 0, nsub = 1;
        if constexpr (kAsym) {
            jg = jt / kT;
            const int r = jt % kT;
            s = r == 0 ? 0 : (r == 1 ? 2 : (r == 2 ? 3 : 1));
            if (r >= 3) { sub = r - 3; nsub = kT - 3; }
        } else if constexpr (kStatBlocks) {
            const int blk = j / NGC;
            jg = j - blk * NGC;
            s = blk == 0 ? 0 : (blk == 1 ? 2 : (blk == 2 ? 1 : 3));
        } else {
            jg = j >> 2;
            s = j & 3;
        }
        const int ri = jg;
        const bool second = s >= 2, is_max = (s & 1) == 0;
        const int sm_ = second ? 1 : 0;
        const GroupWin win = make_win(a, R.P(0, ri), fast_err(R.rkd(0, ri).hi), fast_err(R.rkd(1, ri).hi), R.fmx(0, ri), R.fmn(0, ri), R.fmx(1, ri),
                                      R.fmn(1, ri), R.gmx(ri));
        const CandTest ct = cand_test(win, s, a.omb1);
        const F2 A = R.A(sm_, ri), rkd = R.rkd(sm_, ri);
        const float S = R.S(sm_, ri);
        // the stored k, read again from the record in global memory (E of this
        // CTA overwrites it only after this phase) in the rare float64 case
        const float* kst_at = reinterpret_cast<const float*>(a.meta + g_first + jg) + 2 * sm_ + 1;
        const auto kst = [kst_at]() { return *kst_at; };
        const float beta = second ? a.beta2 : a.beta1, omb = second ? a.omb2 : a.omb1;
        float best = is_max ? 0.0f : kInf;
        uint32_t h = R.holders(s, ri);
        if (nsub > 1) {   // every nsub-th holder lane for this thread of the job
            uint32_t mine = 0u;
            int k = 0;
            for (uint32_t t = h; t; t &= t - 1u, ++k)
                if (k % nsub == sub) mine |= t & (0u - t);
            h = mine;
        }
        while (h) {
            const int ln = __ffs(h) - 1;
            h &= h - 1u;
            const int th = (int)R.hwarp(ri) * 32 + ln;
            float* vals = second ? sm_v[th] : sm_m[th];
            // the holder's gradients and codes, read again from L2 (zero beyond n)
            uint32_t gw[8], cw[4];
            reload_inputs(a, cta_base + (int64_t)th * kVec, second, gw, cw);
            uint32_t msk = 0u;
            if constexpr (kStatBlocks) {
                // the window test of the job's statistic alone (`cand` without its
                // inputs-live clause, which only decides for values exactly zero)
                uint32_t zm = 0u;
                if (is_max) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float4 x = *reinterpret_cast<const float4*>(vals + chunk_slot(th, q));
                        msk |= ((fabsf(x.x) >= ct.hi ? 1u : 0u) | (fabsf(x.y) >= ct.hi ? 2u : 0u) |
                                (fabsf(x.z) >= ct.hi ? 4u : 0u) | (fabsf(x.w) >= ct.hi ? 8u : 0u))
                               << (4 * q);
                    }
                    if (!(ct.hi > 0.0f)) {   // a degenerate window admits zeros
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float4 x = *reinterpret_cast<const float4*>(vals + chunk_slot(th, q));
                            zm |= ((x.x == 0.0f ? 1u : 0u) | (x.y == 0.0f ? 2u : 0u) |
                                   (x.z == 0.0f ? 4u : 0u) | (x.w == 0.0f ? 8u : 0u)) << (4 * q);
                        }
                    }
                } else if (second) {         // v: T_j = v_j, lo = max(a0, 0)
                    const float lo = fmaxf(ct.a0, 0.0f);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float4 x = *reinterpret_cast<const float4*>(vals + chunk_slot(th, q));
                        msk |= ((fabsf(x.x) <= lo ? 1u : 0u) | (fabsf(x.y) <= lo ? 2u : 0u) |
                                (fabsf(x.z) <= lo ? 4u : 0u) | (fabsf(x.w) <= lo ? 8u : 0u)) << (4 * q);
                        zm |= ((x.x == 0.0f ? 1u : 0u) | (x.y == 0.0f ? 2u : 0u) |
                               (x.z == 0.0f ? 4u : 0u) | (x.w == 0.0f ? 8u : 0u)) << (4 * q);
                    }
                } else {                     // m: T_j = |m_j| + 2 (1 - beta1) |g_j|
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const float4 x = *reinterpret_cast<const float4*>(vals + chunk_slot(th, q));
                        const float xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const float ax = fabsf(xs[i]);
                            const float Tj = fmaf(ct.c, fabsf(bf16_of(gw, 4 * q + i)), ax);
                            const float lo = fmaxf(fmaf(ct.a1, Tj, ct.a0), ct.a2 * Tj);
                            msk |= (ax <= lo ? 1u : 0u) << (4 * q + i);
                            zm |= (ax == 0.0f ? 1u : 0u) << (4 * q + i);
                        }
                    }
                }
                // a value of exactly zero is a candidate only when its inputs are
                // not both zero (the moment of zero inputs is exactly zero)
                uint32_t zc = msk & zm;
                while (zc) {
                    const int e = __ffs(zc) - 1;
                    zc &= zc - 1u;
                    if (bf16_of(gw, e) == 0.0f && (byte_of(cw, e) & 0x7Fu) == 0u) msk &= ~(1u << e);
                }
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 x = *reinterpret_cast<const float4*>(vals + chunk_slot(th, q));
                    msk |= (cand(x.x, fabsf(bf16_of(gw, 4 * q)), byte_of(cw, 4 * q), ct) ? 1u : 0u) << (4 * q);
                    msk |= (cand(x.y, fabsf(bf16_of(gw, 4 * q + 1)), byte_of(cw, 4 * q + 1), ct) ? 1u : 0u) << (4 * q + 1);
                    msk |= (cand(x.z, fabsf(bf16_of(gw, 4 * q + 2)), byte_of(cw, 4 * q + 2), ct) ? 1u : 0u) << (4 * q + 2);
                    msk |= (cand(x.w, fabsf(bf16_of(gw, 4 * q + 3)), byte_of(cw, 4 * q + 3), ct) ? 1u : 0u) << (4 * q + 3);
                }
            }
            while (msk) {
                const int e = __ffs(msk) - 1;
                msk &= msk - 1u;
                const float x = exact_moment(byte_of(cw, e), bf16_of(gw, e), second, A, rkd, S,
                                             kst, beta, omb, tab, lg_hi, lg_lo);
                vals[chunk_slot(th, e >> 2) + (e & 3)] = x;   // encoded from the exact value
                const float ax = fabsf(x);
                if (is_max) best = fmaxf(best, ax);
                else if (ax > 0.0f) best = fminf(best, ax);
            }
        }
        if constexpr (kAsym) {
            const int r = jt % kT;
            float mm = r >= 3 ? best : kInf;
#pragma unroll
            for (int off = 1; off < kT; off <<= 1) mm = fminf(mm, __shfl_xor_sync(kFull, mm, off));
            if (r > 3) continue;
            if (r == 3) best = mm;
        }
        best = (best < kInf) ? best : 0.0f;
        R.ex(s, ri) = best;
        R.lex(s, ri) = best > 0.0f ? df::log2_df(best, tab) : F2{0.0f, 0.0f};
    }
    __syncthreads();

    // ---- E: fresh k, S, encoding constants and the group record ----
    for (int j = tid; j < 2 * NGC; j += kCta) {
        const int jg = j >> 1, sm_ = j & 1;
        const int ri = jg;
        const float mx = R.ex(2 * sm_, ri), mn = R.ex(2 * sm_ + 1, ri);
        float k, S;
        k_and_S_logs(mx, mn, R.lex(2 * sm_, ri), R.lex(2 * sm_ + 1, ri), tab, k, S);
        float inv, cz;
        encode_consts(mx, k, inv, cz);
        R.k(sm_, ri) = k;
        R.inv(sm_, ri) = inv;
        R.cz(sm_, ri) = cz;
        const int64_t gg = g_first + jg;
        if (gg * G < a.n) reinterpret_cast<float2*>(a.meta + gg)[sm_] = make_float2(S, k);
    }
    __syncthreads();

    // ---- F: encode and store the codes ----
    if (!active) return;
    {
        const int ri = gi;
        const float km = R.k(0, ri), invm = R.inv(0, ri), czm = R.cz(0, ri);
        const float kv = R.k(1, ri), invv = R.inv(1, ri), czv = R.cz(1, ri);
        uint32_t om[4], ov[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int slot = chunk_slot(tid, q);
            const float4 m4 = *reinterpret_cast<const float4*>(&sm_m[tid][slot]);
            const float4 v4 = *reinterpret_cast<const float4*>(&sm_v[tid][slot]);
            om[q] = e4m3_canonical_zero(encode_pair_m(m4.x, m4.y, km, invm, czm) |
                                        (encode_pair_m(m4.z, m4.w, km, invm, czm) << 16));
            ov[q] = encode_pair_v(v4.x, v4.y, kv, invv, czv) | (encode_pair_v(v4.z, v4.w, kv, invv, czv) << 16);
        }
        if (full) {
            st_cs(reinterpret_cast<uint4*>(a.mq + base), make_uint4(om[0], om[1], om[2], om[3]));
            st_cs(reinterpret_cast<uint4*>(a.vq + base), make_uint4(ov[0], ov[1], ov[2], ov[3]));
        } else {
#pragma unroll
            for (int e = 0; e < kVec; ++e) {
                if (base + e < a.n) {
                    a.mq[base + e] = (uint8_t)(om[e / 4] >> (8 * (e & 3)));
                    a.vq[base + e] = (uint8_t)(ov[e / 4] >> (8 * (e & 3)));
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------
// G < 16: a thread holds 16/G whole groups (the same arithmetic, per thread)
// ---------------------------------------------------------------------------
constexpr int kThreadCta = 128;

template <int G>
__global__ void __launch_bounds__(kThreadCta)
step_kernel_thread(const StepArgs a) {
    constexpr int NG = kVec / G;
    __shared__ float lg_hi[128], lg_lo[128];
    __shared__ SmemTables st;
    for (int i = threadIdx.x; i < 128; i += kThreadCta) {
        lg_hi[i] = __uint_as_float(gtab::kLog2Frac448Hi[i]);
        lg_lo[i] = __uint_as_float(gtab::kLog2Frac448Lo[i]);
    }
    load_smem_tables(st, threadIdx.x, kThreadCta);
    __syncthreads();
    const df::Tables tab = tables_of(st);

    const int64_t base = ((int64_t)blockIdx.x * kThreadCta + threadIdx.x) * kVec;
    if (base >= a.n) return;
    const bool full = base + kVec <= a.n;
    const int64_t g0 = base / G;

    Chunk c;
    load_chunk(a, base, full, c);
    float m[kVec], v[kVec];
    float km[NG], kv[NG], Sm[NG], Sv[NG], inv_m[NG], cz_m[NG], inv_v[NG], cz_v[NG];
#pragma unroll
    for (int j = 0; j < NG; ++j) {
        float4 md = make_float4(0.0f, 1.0f, 0.0f, 1.0f);
        if ((g0 + j) * G < a.n) md = ld_cs(a.meta + g0 + j);
        const StateParams pm = state_params(md.x, md.y, tab);
        const StateParams pv = state_params(md.z, md.w, tab);
        const float eps_m = fast_err(pm.rkd.hi), eps_v = fast_err(pv.rkd.hi);
        float fmx_m = 0.0f, fmx_v = 0.0f, gmx = 0.0f, fmn_m = kInf, fmn_v = kInf;
#pragma unroll
        for (int i = 0; i < G; ++i) {
            const int e = j * G + i;
            const float gf = bf16_of(c.g, e);
            fast_elem<0>(a, byte_of(c.mq, e), byte_of(c.vq, e), gf, c.w[e], lg_hi, a.beta1 * pm.P,
                         pm.rkd.hi, a.beta2 * pv.P, pv.rkd.hi, m[e], v[e]);
            fmx_m = fmaxf(fmx_m, fabsf(m[e]));
            fmx_v = fmaxf(fmx_v, v[e]);
            gmx = fmaxf(gmx, fabsf(gf));
            fmn_m = fminf(fmn_m, nz_key(m[e]));
            fmn_v = fminf(fmn_v, nz_key(v[e]));
        }
        const GroupWin win = make_win(a, pm.P, eps_m, eps_v, fmx_m, nz_key_value(fmn_m), fmx_v,
                                      nz_key_value(fmn_v), gmx);
        float ex[4] = {0.0f, kInf, 0.0f, kInf};
        // every element inside any window is re-evaluated once and encoded exactly
#pragma unroll
        for (int i = 0; i < G; ++i) {
            const int e = j * G + i;
            const float gf = bf16_of(c.g, e);
            const uint32_t cmq = byte_of(c.mq, e), cvq = byte_of(c.vq, e);
            const bool cm = cand(m[e], fabsf(gf), cmq, cand_test(win, 0, a.omb1)) ||
                            cand(m[e], fabsf(gf), cmq, cand_test(win, 1, a.omb1));
            const bool cv = cand(v[e], fabsf(gf), cvq, cand_test(win, 2, a.omb1)) ||
                            cand(v[e], fabsf(gf), cvq, cand_test(win, 3, a.omb1));
            if (cm) {
                m[e] = exact_moment(byte_of(c.mq, e), gf, false, pm.A, pm.rkd, pm.S,
                                    [k = md.y]() { return k; },
                                    a.beta1, a.omb1, tab, lg_hi, lg_lo);
                const float ax = fabsf(m[e]);
                ex[0] = fmaxf(ex[0], ax);
                if (ax > 0.0f) ex[1] = fminf(ex[1], ax);
            }
            if (cv) {
                v[e] = exact_moment(byte_of(c.vq, e), gf, true, pv.A, pv.rkd, pv.S,
                                    [k = md.w]() { return k; },
                                    a.beta2, a.omb2, tab, lg_hi, lg_lo);
                const float ax = fabsf(v[e]);
                ex[2] = fmaxf(ex[2], ax);
                if (ax > 0.0f) ex[3] = fminf(ex[3], ax);
            }
        }
        if (!(ex[1] < kInf)) ex[1] = 0.0f;
        if (!(ex[3] < kInf)) ex[3] = 0.0f;
        k_and_S(ex[0], ex[1], tab, km[j], Sm[j]);
        k_and_S(ex[2], ex[3], tab, kv[j], Sv[j]);
        encode_consts(ex[0], km[j], inv_m[j], cz_m[j]);
        encode_consts(ex[2], kv[j], inv_v[j], cz_v[j]);
    }
    store_w(a, base, full, c);
    uint32_t om[4], ov[4];
#pragma unroll
    for (int e = 0; e < kVec; e += 2) {
        const int j0 = e / G, j1 = (e + 1) / G;
        const float ym0 = copysignf(ex2_ftz(fmaf(km[j0], lg2_ftz(fabsf(m[e]) * inv_m[j0]), cz_m[j0])), m[e]);
        const float ym1 = copysignf(ex2_ftz(fmaf(km[j1], lg2_ftz(fabsf(m[e + 1]) * inv_m[j1]), cz_m[j1])), m[e + 1]);
        const float yv0 = ex2_ftz(fmaf(kv[j0], lg2_ftz(v[e] * inv_v[j0]), cz_v[j0]));
        const float yv1 = ex2_ftz(fmaf(kv[j1], lg2_ftz(v[e + 1] * inv_v[j1]), cz_v[j1]));
        const uint32_t pm_ = e4m3_canonical_zero(e4m3x2(ym0, ym1)), pv_ = e4m3x2(yv0, yv1);
        if ((e & 2) == 0) { om[e / 4] = pm_; ov[e / 4] = pv_; }
        else { om[e / 4] |= pm_ << 16; ov[e / 4] |= pv_ << 16; }
    }
    if (full) {
        st_cs(reinterpret_cast<uint4*>(a.mq + base), make_uint4(om[0], om[1], om[2], om[3]));
        st_cs(reinterpret_cast<uint4*>(a.vq + base), make_uint4(ov[0], ov[1], ov[2], ov[3]));
    } else {
#pragma unroll
        for (int e = 0; e < kVec; ++e) {
            if (base + e < a.n) {
                a.mq[base + e] = (uint8_t)(om[e / 4] >> (8 * (e & 3)));
                a.vq[base + e] = (uint8_t)(ov[e / 4] >> (8 * (e & 3)));
            }
        }
    }
#pragma unroll
    for (int j = 0; j < NG; ++j)
        if ((g0 + j) * G < a.n) st_cs(a.meta + g0 + j, make_float4(Sm[j], km[j], Sv[j], kv[j]));
}

template <int G>
cudaError_t launch_step(const StepArgs& a, cudaStream_t stream) {
    if constexpr (G >= kVec) {
        constexpr int CTA = kStepCta;
        using Lay = CtaLayout<G, CTA>;
        // more than 48 KB of dynamic shared memory needs the opt-in attribute
        const cudaError_t e = cudaFuncSetAttribute(step_kernel_cta<G, CTA>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   (int)Lay::bytes);
        if (e != cudaSuccess) return e;
        const int64_t blocks = (a.n + Lay::kCtaElems - 1) / Lay::kCtaElems;
        step_kernel_cta<G, CTA><<<(unsigned)blocks, CTA, Lay::bytes, stream>>>(a);
    } else {
        const int64_t threads = (a.n + kVec - 1) / kVec;
        const int64_t blocks = (threads + kThreadCta - 1) / kThreadCta;
        step_kernel_thread<G><<<(unsigned)blocks, kThreadCta, 0, stream>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t read_recompute_counts(unsigned long long out[2], bool reset) {
    cudaError_t e = cudaMemcpyFromSymbol(out, g_recompute, sizeof(unsigned long long) * 2);
    if (e == cudaSuccess && reset) {
        const unsigned long long zero[2] = {0ull, 0ull};
        e = cudaMemcpyToSymbol(g_recompute, zero, sizeof(zero));
    }
    return e;
}

cudaError_t launch_adamw_dre_step(const StepArgs& a, int G, cudaStream_t stream) {
    switch (G) {
        case 1: return launch_step<1>(a, stream);
        case 2: return launch_step<2>(a, stream);
        case 4: return launch_step<4>(a, stream);
        case 8: return launch_step<8>(a, stream);
        case 16: return launch_step<16>(a, stream);
        case 32: return launch_step<32>(a, stream);
        case 64: return launch_step<64>(a, stream);
        case 128: return launch_step<128>(a, stream);
        case 256: return launch_step<256>(a, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace coat
