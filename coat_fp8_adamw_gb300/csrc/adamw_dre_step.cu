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
// first computed on a fast fp32/SFU path whose error is bounded (kFastErr);
// the elements whose fast value lies within twice that bound of the group's
// fast max (min) are re-evaluated exactly -- (|E4M3(q)| S)^(1/k) in
// double-float, rounded once, then beta x + (1 - beta) g as a correctly
// rounded sum of two products -- and the group's max and min are taken over
// those exact values.  k and S are formed from them in double-float and
// rounded once.  All codes are encoded from the fast values and the exact
// (max, k).
//
// Layout: every thread owns 16 consecutive parameters, so each stream is
// whole 128-bit accesses: w 4x16 B, g 2x16 B, m codes 16 B, v codes 16 B;
// the 16-byte (S_m, k_m, S_v, k_v) record per group is one 128-bit access.
// For G >= 32 a group spans G/16 adjacent lanes of a warp and the per-group
// work is split across them; for G <= 16 a thread holds 16/G whole groups.
#include <cstddef>

#include "coat_device.cuh"
#include "coat_kernels.h"

namespace coat {

namespace {

using df::F2;

constexpr int kStepThreads = 128;   // 4 warps per CTA
constexpr unsigned kFull = 0xFFFFFFFFu;

// Bound on the relative error of a fast dequantized moment (SFU exp2 2^-22,
// the fp32 exponent L(q)/k with |L(q)/k| <= 277 rounded three times, P a few
// ulp, two roundings) with ample margin.  Through the EMA it bounds the error
// of v_t relative to v_t and of m_t relative to |beta1 m| + |(1-beta1) g|.
constexpr float kFastErr = 6.103515625e-05f;   // 2^-14

template <int G>
struct Geom {
    static constexpr int kLanes = G >= kVec ? G / kVec : 1;   // lanes per group
    static constexpr int kGroups = G >= kVec ? 1 : kVec / G;  // groups per thread
    static constexpr int kElems = G >= kVec ? kVec : G;       // elements per (thread, group)
};

// Per-warp staging: the fast moments and the raw inputs of every lane, read
// by the lanes that look for and re-evaluate a group's extreme elements.
// Row strides (20 and 12 words) keep the 128-bit stores bank-conflict free;
// every row starts on a 16-byte boundary (128-bit shared-memory stores).
struct alignas(16) WarpStage {
    float m[32][20];
    float v[32][20];
    uint32_t mq[32][4];
    uint32_t vq[32][4];
    uint32_t g[32][12];
};

struct StepSmem {
    WarpStage stage[kStepThreads / 32];   // first: 16-byte aligned at offset 0
    float lg_hi[128];
    float lg_lo[128];
    SmemTables t;
};
static_assert(offsetof(StepSmem, stage) % 16 == 0, "staging must be 16-byte aligned");
static_assert(sizeof(WarpStage) % 16 == 0, "per-warp staging must keep 16-byte alignment");
static_assert(offsetof(WarpStage, m) % 16 == 0 && offsetof(WarpStage, v) % 16 == 0 &&
              offsetof(WarpStage, mq) % 16 == 0 && offsetof(WarpStage, vq) % 16 == 0 &&
              offsetof(WarpStage, g) % 16 == 0, "rows of 128-bit stores");
static_assert((20 * 4) % 16 == 0 && (12 * 4) % 16 == 0 && (4 * 4) % 16 == 0, "row strides");

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
        const uint4* gp = reinterpret_cast<const uint4*>(a.g + base);
        const uint4 g0 = ld_cs(gp), g1 = ld_cs(gp + 1);
        c.g[0] = g0.x; c.g[1] = g0.y; c.g[2] = g0.z; c.g[3] = g0.w;
        c.g[4] = g1.x; c.g[5] = g1.y; c.g[6] = g1.z; c.g[7] = g1.w;
        const uint4 m = ld_cs(reinterpret_cast<const uint4*>(a.mq + base));
        const uint4 v = ld_cs(reinterpret_cast<const uint4*>(a.vq + base));
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

__device__ __forceinline__ void zero_chunk(Chunk& c) {
#pragma unroll
    for (int e = 0; e < kVec; ++e) c.w[e] = 0.0f;
#pragma unroll
    for (int i = 0; i < kVec / 2; ++i) c.g[i] = 0u;
#pragma unroll
    for (int i = 0; i < kVec / 4; ++i) { c.mq[i] = 0u; c.vq[i] = 0u; }
}

__device__ __forceinline__ uint32_t byte_of(const uint32_t* w, int j) {
    return (w[j >> 2] >> (8 * (j & 3))) & 0xFFu;
}
__device__ __forceinline__ float bf16_of(const uint32_t* w, int j) {
    return (j & 1) ? __uint_as_float(w[j >> 1] & 0xFFFF0000u) : __uint_as_float(w[j >> 1] << 16);
}

// Parameters of one stored moment.  Exact path: A = log2(448 S) and 1/k as
// double-floats.  Fast path: P = (448 S)^(1/k) and 1/k as floats.
struct StateParams {
    F2 A;
    F2 rkd;
    float P;
};

__device__ __forceinline__ StateParams state_params(float S, float k, const df::Tables& t) {
    StateParams p;
    p.rkd = df::div21(F2{1.0f, 0.0f}, k);
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
__device__ __forceinline__ float exact_moment(uint32_t code, float gf, bool second,
                                              const StateParams& sp, float beta, float omb,
                                              const df::Tables& t, const float* lg_hi,
                                              const float* lg_lo) {
    float prev = 0.0f;
    const uint32_t mag = code & 0x7Fu;
    if (mag != 0u && sp.P > 0.0f) {
        const F2 L = {lg_hi[mag], lg_lo[mag]};
        prev = df::exp2_df(df::mul22(df::add2(L, sp.A), sp.rkd), t);
        if (code & 0x80u) prev = -prev;
    }
    const float x = second ? __fmul_rn(gf, gf) : gf;
    return df::dot2_rn(beta, prev, omb, x);
}

// k rounded once from double-float logs of the group's max / min magnitudes,
// with the cap and the S-range guard; S = 2^(k log2 max - log2 448) rounded once.
__device__ __forceinline__ void k_and_S(float mx, float mn, F2 Lmx, F2 Lmn, const df::Tables& t,
                                        float& k, float& S) {
    if (!(mx > 0.0f)) {
        k = 1.0f;
        S = 0.0f;
        return;
    }
    k = 1.0f;
    if (mn > 0.0f && mn < mx)
        k = fminf(df::div22_rn(const_df(kLog2RDf), df::add2(Lmx, df::neg2(Lmn))), kKCap);
    if (Lmx.hi < 0.0f)
        k = fminf(k, df::div22_rn(const_df(kGuardLoDf), Lmx));
    else if (Lmx.hi > 0.0f)
        k = fminf(k, df::div22_rn(const_df(kGuardHiDf), Lmx));
    S = df::exp2_df(df::add2(df::mul21(Lmx, k), df::neg2(const_df(kLog2_448Df))), t);
}

// Encoding constants of one group: r = |x| * inv, z = k log2 r + cz.  A
// subnormal max is pre-scaled by 2^24 (inv = 1/(max 2^24)) and the factor is
// folded back into cz.
struct EncodeParams {
    float inv;
    float k;
    float cz;
};

__device__ __forceinline__ EncodeParams encode_params(float mx, float k) {
    EncodeParams e;
    e.k = k;
    const bool sub = mx < 1.17549435e-38f;
    e.inv = mx > 0.0f ? __frcp_rn(sub ? mx * 16777216.0f : mx) : 0.0f;
    e.cz = sub ? fmaf(24.0f, k, kLog2_448) : kLog2_448;
    return e;
}

// Smallest-non-zero keys: 2 * bits(|x|) - 2 as unsigned drops the sign and
// sends +-0 to 0xFFFFFFFE, above every non-zero magnitude.
__device__ __forceinline__ uint32_t min_key(float x) { return __float_as_uint(x) * 2u - 2u; }
__device__ __forceinline__ float min_key_value(uint32_t k) {
    return k >= 0xFFFFFFFEu ? 0.0f : __uint_as_float((k + 2u) >> 1);
}

// ---------------------------------------------------------------------------
// the fast path over one thread's 16 elements (shared by both kernels)
// ---------------------------------------------------------------------------
template <int NG, int E>
__device__ __forceinline__ void fast_path(const StepArgs& a, Chunk& c, const float* lg,
                                          const float* Pm, const float* rkm, const float* Pv,
                                          const float* rkv, float* m, float* v, float* mx_m,
                                          uint32_t* mn_m, float* mx_v, uint32_t* mn_v,
                                          float* mx_g) {
#pragma unroll
    for (int j = 0; j < NG; ++j) {
        mx_m[j] = 0.0f; mx_v[j] = 0.0f; mx_g[j] = 0.0f; mn_m[j] = 0xFFFFFFFEu; mn_v[j] = 0xFFFFFFFEu;
    }
#pragma unroll
    for (int e = 0; e < kVec; ++e) {
        const int j = e / E;
        const uint32_t wm = c.mq[e / 4] >> (8 * (e & 3));
        const uint32_t wv = c.vq[e / 4] >> (8 * (e & 3));
        // dequantize: |x| = P 2^(L(q)/k); the code's sign goes onto P, and the
        // "+ 0" keeps a zero magnitude at +0 whatever the sign bit
        const float em = ex2_ftz(__fmul_rn(lg[wm & 0x7Fu], rkm[j]));
        const float Ps = __uint_as_float(__float_as_uint(Pm[j]) | ((wm & 0x80u) << 24));
        const float m_prev = fmaf(em, Ps, 0.0f);
        const float v_prev = __fmul_rn(Pv[j], ex2_ftz(__fmul_rn(lg[wv & 0x7Fu], rkv[j])));
        const float gf = bf16_of(c.g, e);
        const float mt = fmaf(a.beta1, m_prev, __fmul_rn(a.omb1, gf));
        const float vt = fmaf(a.beta2, v_prev, __fmul_rn(__fmul_rn(a.omb2, gf), gf));
        // AdamW; sqrt/rcp on the SFU (flush-to-zero only below 2^-126)
        const float denom = __fadd_rn(sqrt_ftz(__fmul_rn(vt, a.c2)), a.eps);
        c.w[e] = fmaf(__fmul_rn(-a.c1, mt), rcp_ftz(denom), __fmul_rn(c.w[e], a.decay));
        m[e] = mt;
        v[e] = vt;
        mx_m[j] = fmaxf(mx_m[j], fabsf(mt));
        mx_v[j] = fmaxf(mx_v[j], vt);
        mx_g[j] = fmaxf(mx_g[j], fabsf(gf));
        mn_m[j] = min(mn_m[j], min_key(mt));
        mn_v[j] = min(mn_v[j], min_key(vt));
    }
}

// Encode 16 moments and store weights, codes.
template <int NG, int E>
__device__ __forceinline__ void encode_store(const StepArgs& a, int64_t base, bool full,
                                             const Chunk& c, const float* m, const float* v,
                                             const EncodeParams* em, const EncodeParams* ev) {
    uint32_t om[kVec / 4], ov[kVec / 4];
#pragma unroll
    for (int e = 0; e < kVec; e += 2) {
        const int j0 = e / E, j1 = (e + 1) / E;
        const float ym0 = copysignf(ex2_ftz(fmaf(em[j0].k, lg2_ftz(fabsf(m[e]) * em[j0].inv), em[j0].cz)), m[e]);
        const float ym1 = copysignf(ex2_ftz(fmaf(em[j1].k, lg2_ftz(fabsf(m[e + 1]) * em[j1].inv), em[j1].cz)), m[e + 1]);
        const float yv0 = ex2_ftz(fmaf(ev[j0].k, lg2_ftz(v[e] * ev[j0].inv), ev[j0].cz));
        const float yv1 = ex2_ftz(fmaf(ev[j1].k, lg2_ftz(v[e + 1] * ev[j1].inv), ev[j1].cz));
        const uint32_t pm = e4m3x2(ym0, ym1);
        const uint32_t pv = e4m3x2(yv0, yv1);
        if ((e & 2) == 0) { om[e / 4] = pm; ov[e / 4] = pv; }
        else { om[e / 4] |= pm << 16; ov[e / 4] |= pv << 16; }
    }
    if (full) {
        float4* wp = reinterpret_cast<float4*>(a.w + base);
#pragma unroll
        for (int i = 0; i < 4; ++i)
            st_cs(wp + i, make_float4(c.w[4 * i], c.w[4 * i + 1], c.w[4 * i + 2], c.w[4 * i + 3]));
        st_cs(reinterpret_cast<uint4*>(a.mq + base), make_uint4(om[0], om[1], om[2], om[3]));
        st_cs(reinterpret_cast<uint4*>(a.vq + base), make_uint4(ov[0], ov[1], ov[2], ov[3]));
    } else {
#pragma unroll
        for (int e = 0; e < kVec; ++e) {
            if (base + e < a.n) {
                a.w[base + e] = c.w[e];
                a.mq[base + e] = (uint8_t)(om[e / 4] >> (8 * (e & 3)));
                a.vq[base + e] = (uint8_t)(ov[e / 4] >> (8 * (e & 3)));
            }
        }
    }
}

// Candidate windows around a group's fast extremes (see kFastErr).
struct Windows {
    float hi_m, lo_m, hi_v, lo_v;   // |m| >= hi_m, 0 < |m| <= lo_m, v >= hi_v, 0 < v <= lo_v
};

__device__ __forceinline__ Windows windows(const StepArgs& a, float P_m, float mx_m, float mn_m,
                                           float mx_v, float mn_v, float mx_g) {
    // m_t may cancel: its error is bounded by kFastErr (beta1 max|m_prev| + (1-beta1) max|g|)
    const float dm = 2.0f * kFastErr * fmaf(a.beta1, P_m * (1.0f + kFastErr), a.omb1 * mx_g);
    Windows w;
    w.hi_m = mx_m - dm;
    w.lo_m = mn_m > 0.0f ? mn_m + dm : -1.0f;
    w.hi_v = mx_v * (1.0f - 2.0f * kFastErr);
    w.lo_v = mn_v > 0.0f ? mn_v * (1.0f + 4.0f * kFastErr) : -1.0f;
    return w;
}

__device__ __forceinline__ bool in_window(float x, int s, const Windows& w) {
    const float ax = fabsf(x);
    switch (s) {
        case 0: return ax >= w.hi_m && ax > 0.0f;
        case 1: return ax <= w.lo_m && ax > 0.0f;
        case 2: return ax >= w.hi_v && ax > 0.0f;
        default: return ax <= w.lo_v && ax > 0.0f;
    }
}

// ---------------------------------------------------------------------------
// G >= 32: a group spans L = G/16 lanes
// ---------------------------------------------------------------------------
template <int G>
__global__ void __launch_bounds__(kStepThreads)
step_kernel_lanes(const StepArgs a) {
    constexpr int L = G / kVec;
    static_assert(L >= 2 && L <= 32, "lanes per group");
    __shared__ StepSmem sm;
    if (threadIdx.x < 128) {
        sm.lg_hi[threadIdx.x] = __uint_as_float(kLog2Frac448Hi[threadIdx.x]);
        sm.lg_lo[threadIdx.x] = __uint_as_float(kLog2Frac448Lo[threadIdx.x]);
    }
    load_smem_tables(sm.t, threadIdx.x, kStepThreads);
    __syncthreads();
    const df::Tables tab = tables_of(sm.t);

    const int lane = threadIdx.x & 31;
    WarpStage& ws = sm.stage[threadIdx.x >> 5];
    const int64_t base = ((int64_t)blockIdx.x * kStepThreads + threadIdx.x) * kVec;
    if (__all_sync(kFull, base >= a.n)) return;   // warp-uniform exit
    const bool active = base < a.n;
    const bool full = base + kVec <= a.n;
    const int64_t grp = base / G;
    const bool group_exists = grp * G < a.n;
    const int lig = lane % L;          // lane within the group
    const int gbase = lane - lig;      // first lane of the group

    Chunk c;
    if (active) load_chunk(a, base, full, c);
    else zero_chunk(c);

    // -- stored-state parameters: even lanes the first moment, odd lanes the second --
    StateParams pm, pv;
    {
        float4 md = make_float4(0.0f, 1.0f, 0.0f, 1.0f);
        if (group_exists) md = ld_cs(a.meta + grp);
        const bool odd = lane & 1;
        const StateParams p = state_params(odd ? md.z : md.x, odd ? md.w : md.y, tab);
        const int sm_ = lane & ~1, sv_ = lane | 1;
        pm.A.hi = __shfl_sync(kFull, p.A.hi, sm_);
        pm.A.lo = __shfl_sync(kFull, p.A.lo, sm_);
        pm.rkd.hi = __shfl_sync(kFull, p.rkd.hi, sm_);
        pm.rkd.lo = __shfl_sync(kFull, p.rkd.lo, sm_);
        pm.P = __shfl_sync(kFull, p.P, sm_);
        pv.A.hi = __shfl_sync(kFull, p.A.hi, sv_);
        pv.A.lo = __shfl_sync(kFull, p.A.lo, sv_);
        pv.rkd.hi = __shfl_sync(kFull, p.rkd.hi, sv_);
        pv.rkd.lo = __shfl_sync(kFull, p.rkd.lo, sv_);
        pv.P = __shfl_sync(kFull, p.P, sv_);
    }

    // -- fast path + stage-1 statistics --
    float m[kVec], v[kVec];
    float lmx_m, lmx_v, lmx_g;
    uint32_t lmn_m, lmn_v;
    fast_path<1, kVec>(a, c, sm.lg_hi, &pm.P, &pm.rkd.hi, &pv.P, &pv.rkd.hi, m, v, &lmx_m, &lmn_m,
                       &lmx_v, &lmn_v, &lmx_g);

    // publish the fast moments and raw inputs of this lane
    {
        float4* pm4 = reinterpret_cast<float4*>(ws.m[lane]);
        float4* pv4 = reinterpret_cast<float4*>(ws.v[lane]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            pm4[i] = make_float4(m[4 * i], m[4 * i + 1], m[4 * i + 2], m[4 * i + 3]);
            pv4[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
        }
        *reinterpret_cast<uint4*>(ws.mq[lane]) = make_uint4(c.mq[0], c.mq[1], c.mq[2], c.mq[3]);
        *reinterpret_cast<uint4*>(ws.vq[lane]) = make_uint4(c.vq[0], c.vq[1], c.vq[2], c.vq[3]);
        *reinterpret_cast<uint4*>(&ws.g[lane][0]) = make_uint4(c.g[0], c.g[1], c.g[2], c.g[3]);
        *reinterpret_cast<uint4*>(&ws.g[lane][4]) = make_uint4(c.g[4], c.g[5], c.g[6], c.g[7]);
    }

    // -- stage 2: across the lanes of the group --
    float mx_m = lmx_m, mx_v = lmx_v, mx_g = lmx_g;
    uint32_t mn_m = lmn_m, mn_v = lmn_v;
#pragma unroll
    for (int off = L / 2; off > 0; off >>= 1) {
        mx_m = fmaxf(mx_m, __shfl_xor_sync(kFull, mx_m, off));
        mx_v = fmaxf(mx_v, __shfl_xor_sync(kFull, mx_v, off));
        mx_g = fmaxf(mx_g, __shfl_xor_sync(kFull, mx_g, off));
        mn_m = min(mn_m, __shfl_xor_sync(kFull, mn_m, off));
        mn_v = min(mn_v, __shfl_xor_sync(kFull, mn_v, off));
    }
    const Windows win = windows(a, pm.P, mx_m, min_key_value(mn_m), mx_v, min_key_value(mn_v), mx_g);

    // lanes whose local extreme falls in a window hold candidates
    const uint32_t gmask = (L == 32) ? kFull : (((1u << L) - 1u) << gbase);
    uint32_t holders[4];
    holders[0] = __ballot_sync(kFull, in_window(lmx_m, 0, win)) & gmask;
    holders[1] = __ballot_sync(kFull, in_window(min_key_value(lmn_m), 1, win)) & gmask;
    holders[2] = __ballot_sync(kFull, in_window(lmx_v, 2, win)) & gmask;
    holders[3] = __ballot_sync(kFull, in_window(min_key_value(lmn_v), 3, win)) & gmask;
    __syncwarp();

    // -- exact extremes: lane lig of the group evaluates the statistics s = lig (mod L) --
    // s: 0 max|m|, 1 smallest non-zero |m|, 2 max v, 3 smallest non-zero v
    float ex[4];
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        const bool is_max = (s & 1) == 0;
        const bool second = s >= 2;
        float best = is_max ? 0.0f : __int_as_float(0x7F800000);
        if (s % L == lig) {
            const StateParams& sp = second ? pv : pm;
            uint32_t h = holders[s];
            while (h) {
                const int lc = __ffs(h) - 1;
                h &= h - 1u;
                const float* vals = second ? ws.v[lc] : ws.m[lc];
                for (int e = 0; e < kVec; ++e) {
                    if (!in_window(vals[e], s, win)) continue;
                    const uint32_t code = byte_of(second ? ws.vq[lc] : ws.mq[lc], e);
                    const float x = fabsf(exact_moment(code, bf16_of(ws.g[lc], e), second, sp,
                                                       second ? a.beta2 : a.beta1,
                                                       second ? a.omb2 : a.omb1, tab, sm.lg_hi,
                                                       sm.lg_lo));
                    if (is_max) best = fmaxf(best, x);
                    else if (x > 0.0f) best = fminf(best, x);
                }
            }
        }
        ex[s] = best;
    }
    __syncwarp();
#pragma unroll
    for (int s = 0; s < 4; ++s) ex[s] = __shfl_sync(kFull, ex[s], gbase + s % L);
    if (!(ex[1] < __int_as_float(0x7F800000))) ex[1] = 0.0f;
    if (!(ex[3] < __int_as_float(0x7F800000))) ex[3] = 0.0f;

    // -- fresh (k, S): even lanes the first moment, odd lanes the second --
    float k_m, S_m, k_v, S_v;
    {
        const bool odd = lane & 1;
        const float mx = odd ? ex[2] : ex[0];
        const float mn = odd ? ex[3] : ex[1];
        const F2 Lmx = mx > 0.0f ? df::log2_df(mx, tab) : F2{0.0f, 0.0f};
        const F2 Lmn = (mn > 0.0f && mn < mx) ? df::log2_df(mn, tab) : F2{0.0f, 0.0f};
        float kk, SS;
        k_and_S(mx, mn, Lmx, Lmn, tab, kk, SS);
        k_m = __shfl_sync(kFull, kk, lane & ~1);
        S_m = __shfl_sync(kFull, SS, lane & ~1);
        k_v = __shfl_sync(kFull, kk, lane | 1);
        S_v = __shfl_sync(kFull, SS, lane | 1);
    }
    if (!active) return;

    const EncodeParams em = encode_params(ex[0], k_m);
    const EncodeParams ev = encode_params(ex[2], k_v);
    encode_store<1, kVec>(a, base, full, c, m, v, &em, &ev);
    if (lig == 0) st_cs(a.meta + grp, make_float4(S_m, k_m, S_v, k_v));
}

// ---------------------------------------------------------------------------
// G <= 16: a thread holds 16/G whole groups
// ---------------------------------------------------------------------------
template <int G>
__global__ void __launch_bounds__(kStepThreads)
step_kernel_thread(const StepArgs a) {
    constexpr int NG = kVec / G;
    constexpr int E = G;
    __shared__ float lg_hi[128], lg_lo[128];
    __shared__ SmemTables st;
    if (threadIdx.x < 128) {
        lg_hi[threadIdx.x] = __uint_as_float(kLog2Frac448Hi[threadIdx.x]);
        lg_lo[threadIdx.x] = __uint_as_float(kLog2Frac448Lo[threadIdx.x]);
    }
    load_smem_tables(st, threadIdx.x, kStepThreads);
    __syncthreads();
    const df::Tables tab = tables_of(st);

    const int64_t base = ((int64_t)blockIdx.x * kStepThreads + threadIdx.x) * kVec;
    if (base >= a.n) return;
    const bool full = base + kVec <= a.n;
    const int64_t g0 = base / G;

    Chunk c;
    load_chunk(a, base, full, c);
    StateParams pm[NG], pv[NG];
    float Pm[NG], Pv[NG], rkm[NG], rkv[NG];
#pragma unroll
    for (int j = 0; j < NG; ++j) {
        float4 md = make_float4(0.0f, 1.0f, 0.0f, 1.0f);
        if ((g0 + j) * G < a.n) md = ld_cs(a.meta + g0 + j);
        pm[j] = state_params(md.x, md.y, tab);
        pv[j] = state_params(md.z, md.w, tab);
        Pm[j] = pm[j].P; rkm[j] = pm[j].rkd.hi; Pv[j] = pv[j].P; rkv[j] = pv[j].rkd.hi;
    }
    float m[kVec], v[kVec];
    float mx_m[NG], mx_v[NG], mx_g[NG];
    uint32_t mn_m[NG], mn_v[NG];
    fast_path<NG, E>(a, c, lg_hi, Pm, rkm, Pv, rkv, m, v, mx_m, mn_m, mx_v, mn_v, mx_g);

    EncodeParams em[NG], ev[NG];
    float k_m[NG], S_m[NG], k_v[NG], S_v[NG];
#pragma unroll
    for (int j = 0; j < NG; ++j) {
        const Windows win = windows(a, Pm[j], mx_m[j], min_key_value(mn_m[j]), mx_v[j],
                                    min_key_value(mn_v[j]), mx_g[j]);
        float ex[4];
#pragma unroll
        for (int s = 0; s < 4; ++s) {
            const bool is_max = (s & 1) == 0;
            const bool second = s >= 2;
            float best = is_max ? 0.0f : __int_as_float(0x7F800000);
#pragma unroll
            for (int ee = 0; ee < E; ++ee) {
                const int e = j * E + ee;
                if (!in_window(second ? v[e] : m[e], s, win)) continue;
                const float x = fabsf(exact_moment(byte_of(second ? c.vq : c.mq, e), bf16_of(c.g, e),
                                                   second, second ? pv[j] : pm[j],
                                                   second ? a.beta2 : a.beta1,
                                                   second ? a.omb2 : a.omb1, tab, lg_hi, lg_lo));
                if (is_max) best = fmaxf(best, x);
                else if (x > 0.0f) best = fminf(best, x);
            }
            ex[s] = best;
        }
        if (!(ex[1] < __int_as_float(0x7F800000))) ex[1] = 0.0f;
        if (!(ex[3] < __int_as_float(0x7F800000))) ex[3] = 0.0f;
#pragma unroll
        for (int st2 = 0; st2 < 2; ++st2) {
            const float mx = ex[2 * st2], mn = ex[2 * st2 + 1];
            const F2 Lmx = mx > 0.0f ? df::log2_df(mx, tab) : F2{0.0f, 0.0f};
            const F2 Lmn = (mn > 0.0f && mn < mx) ? df::log2_df(mn, tab) : F2{0.0f, 0.0f};
            if (st2 == 0) k_and_S(mx, mn, Lmx, Lmn, tab, k_m[j], S_m[j]);
            else k_and_S(mx, mn, Lmx, Lmn, tab, k_v[j], S_v[j]);
        }
        em[j] = encode_params(ex[0], k_m[j]);
        ev[j] = encode_params(ex[2], k_v[j]);
    }
    encode_store<NG, E>(a, base, full, c, m, v, em, ev);
#pragma unroll
    for (int j = 0; j < NG; ++j)
        if ((g0 + j) * G < a.n) st_cs(a.meta + g0 + j, make_float4(S_m[j], k_m[j], S_v[j], k_v[j]));
}

template <int G>
cudaError_t launch_step(const StepArgs& a, cudaStream_t stream) {
    const int64_t threads = (a.n + kVec - 1) / kVec;
    const int64_t blocks = (threads + kStepThreads - 1) / kStepThreads;
    if constexpr (G >= 2 * kVec)
        step_kernel_lanes<G><<<(unsigned)blocks, kStepThreads, 0, stream>>>(a);
    else
        step_kernel_thread<G><<<(unsigned)blocks, kStepThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

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
