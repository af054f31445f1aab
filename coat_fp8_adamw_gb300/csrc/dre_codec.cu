// dre_codec.cu -- standalone Dynamic Range Expansion quantizer / dequantizer
// for one fp32 tensor (COAT paper-review page, section 3: FP8 quantization
// equation and the Dynamic Range Expansion equations).  Same thread layout and
// per-group arithmetic as the fused step: 16 elements per thread, a group of
// G >= 16 spans G/16 adjacent lanes, two-stage max / smallest-non-zero
// reduction (per thread, then warp shuffles).
#include "coat_kernels.h"
#include "coat_device.cuh"

namespace coat {

namespace {

template <int G>
struct Geom {
    static constexpr int kLanes = G >= kVec ? G / kVec : 1;
    static constexpr int kGroups = G >= kVec ? 1 : kVec / G;
    static constexpr int kElems = G >= kVec ? kVec : G;
    // several lanes share a group: its parameters are formed once per CTA job
    static constexpr bool kJobs = G >= 2 * kVec;
    static constexpr int kGpc = kJobs ? kThreads * kVec / G : 1;   // groups per CTA
};

// The per-group shared arrays of the job form (G >= 32).
template <int N>
struct QuantJobs {
    float mx[N], k[N], inv[N], pre[N];
    uint32_t mn[N];
};

// One thread's 16 values x of the tile starting at element `base`: group
// statistics, k and S (formed once per group of the CTA in the job form),
// codes stored, and the group records written.  Every thread of the CTA
// calls it (the job form has CTA barriers).
template <int G>
__device__ __forceinline__ void quantize_tile(const QuantArgs& a, const float (&x)[kVec], int64_t base,
                                              int64_t cta_group0, const df::Tables& tab,
                                              QuantJobs<Geom<G>::kGpc>& sj) {
    using Gm = Geom<G>;
    const bool active = base < a.n;
    const bool full = base + kVec <= a.n;
    float mx[Gm::kGroups];
    uint32_t mn[Gm::kGroups];
#pragma unroll
    for (int j = 0; j < Gm::kGroups; ++j) { mx[j] = 0.0f; mn[j] = 0xFFFFFFFFu; }
#pragma unroll
    for (int e = 0; e < kVec; ++e) {
        const int j = e / Gm::kElems;
        const float ax = fabsf(x[e]);
        mx[j] = fmaxf(mx[j], ax);
        mn[j] = min(mn[j], nz_key(ax));
    }
#pragma unroll
    for (int off = Gm::kLanes / 2; off > 0; off >>= 1) {
        mx[0] = fmaxf(mx[0], __shfl_xor_sync(0xFFFFFFFFu, mx[0], off));
        mn[0] = min(mn[0], __shfl_xor_sync(0xFFFFFFFFu, mn[0], off));
    }
    QuantParams qp[Gm::kGroups];
    float pre[Gm::kGroups];
    if constexpr (Gm::kJobs) {
        // one thread per group of the CTA forms k, S and the encoding
        // constants (the lanes of a group would otherwise each repeat them)
        const int gl = (int)((threadIdx.x * kVec) / G);
        if ((threadIdx.x * kVec) % G == 0) {
            sj.mx[gl] = mx[0];
            sj.mn[gl] = mn[0];
        }
        __syncthreads();
        // With a warp or less of jobs (G >= 128) two adjacent lanes take a
        // group: each forms one of the two logs (max, smallest non-zero), so
        // that their chains run side by side, and the even lane takes the
        // other's by a shuffle and forms k, S and the rest (1-3 % faster; with
        // more jobs the extra lanes cost more than the overlap saves).
        constexpr int kPer = Gm::kGpc <= 32 ? 2 : 1;
        static_assert(kPer == 1 || (2 * Gm::kGpc) % 32 == 0, "whole warps of job lanes");
        for (int j2 = threadIdx.x; j2 < kPer * Gm::kGpc; j2 += kThreads) {
            const int j = j2 / kPer;
            const float gm = sj.mx[j], gmn = nz_key_value(sj.mn[j]);
            QuantParams q;
            if constexpr (kPer == 2) {
                const bool lmin = (j2 & 1) != 0;
                const float arg = lmin && gmn > 0.0f && gmn < gm ? gmn : gm;
                const df::F2 L = gm > 0.0f ? df::log2_df(arg, tab) : df::F2{0.0f, 0.0f};
                const df::F2 Lo = {__shfl_xor_sync(0xFFFFFFFFu, L.hi, 1), __shfl_xor_sync(0xFFFFFFFFu, L.lo, 1)};
                if (lmin) continue;
                q = quant_params_logs(gm, gmn, L, Lo, tab);
            } else {
                q = quant_params_precise(gm, gmn, tab);
            }
            float pr = 1.0f;
            if (gm > 0.0f && gm < 1.17549435e-38f) {
                pr = 16777216.0f;
                q.inv_mx = __frcp_rn(gm * 16777216.0f);
            }
            sj.k[j] = q.k;
            sj.inv[j] = q.inv_mx;
            sj.pre[j] = pr;
            if ((cta_group0 + j) * G < a.n) {
                a.scale[cta_group0 + j] = q.S;
                a.k[cta_group0 + j] = q.k;
            }
        }
        __syncthreads();
        qp[0].k = sj.k[gl];
        qp[0].inv_mx = sj.inv[gl];
        pre[0] = sj.pre[gl];
    } else {
#pragma unroll
        for (int j = 0; j < Gm::kGroups; ++j) {
            qp[j] = quant_params_precise(mx[j], nz_key_value(mn[j]), tab);
            pre[j] = 1.0f;
            if (mx[j] > 0.0f && mx[j] < 1.17549435e-38f) {
                pre[j] = 16777216.0f;
                qp[j].inv_mx = __frcp_rn(mx[j] * 16777216.0f);
            }
        }
    }
    if (!active) return;

    uint32_t out[kVec / 4];
#pragma unroll
    for (int e = 0; e < kVec; e += 2) {
        const int j0 = e / Gm::kElems, j1 = (e + 1) / Gm::kElems;
        const float r0 = (fabsf(x[e]) * pre[j0]) * qp[j0].inv_mx;
        const float r1 = (fabsf(x[e + 1]) * pre[j1]) * qp[j1].inv_mx;
        const uint32_t p = e4m3x2(expand_scaled(x[e], r0, qp[j0].k), expand_scaled(x[e + 1], r1, qp[j1].k));
        if ((e & 2) == 0) out[e / 4] = p; else out[e / 4] |= p << 16;
    }
#pragma unroll
    for (int i = 0; i < kVec / 4; ++i) out[i] = e4m3_canonical_zero(out[i]);
    if (full) {
        st_cs(reinterpret_cast<uint4*>(a.q + base), make_uint4(out[0], out[1], out[2], out[3]));
    } else {
#pragma unroll
        for (int e = 0; e < kVec; ++e)
            if (base + e < a.n) a.q[base + e] = (uint8_t)(out[e / 4] >> (8 * (e & 3)));
    }
    if constexpr (!Gm::kJobs) {
        const int64_t g0 = base / G;
        const bool leader = G >= kVec ? ((base % G) == 0) : true;
        if (leader) {
#pragma unroll
            for (int j = 0; j < Gm::kGroups; ++j)
                if ((g0 + j) * G < a.n) { a.scale[g0 + j] = qp[j].S; a.k[g0 + j] = qp[j].k; }
        }
    }
}

// One tile of 4096 elements per CTA.  Eight 256-thread CTAs per SM for
// G >= 16 (32 registers, a few spilled): the kernel is latency-bound and
// occupancy pays more than the spills cost; below G = 16 a thread holds 16/G
// groups and the register need grows with them.
template <int G>
__global__ void __launch_bounds__(kThreads, G >= kVec ? 8 : 1)
dre_quantize_kernel(const QuantArgs a) {
    __shared__ SmemTables st;
    __shared__ QuantJobs<Geom<G>::kGpc> sj;
    const int64_t base = ((int64_t)blockIdx.x * kThreads + threadIdx.x) * kVec;
    // the inputs first: their loads are in flight while the tables are filled
    float x[kVec];
    if (base + kVec <= a.n) {
        const float4* xp = reinterpret_cast<const float4*>(a.x + base);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 t = ld_cs(xp + i);
            x[4 * i] = t.x; x[4 * i + 1] = t.y; x[4 * i + 2] = t.z; x[4 * i + 3] = t.w;
        }
    } else {
#pragma unroll
        for (int e = 0; e < kVec; ++e) x[e] = base + e < a.n ? a.x[base + e] : 0.0f;
    }
    load_smem_tables(st, threadIdx.x, kThreads);
    __syncthreads();
    if (!Geom<G>::kJobs && __all_sync(0xFFFFFFFFu, base >= a.n)) return;
    quantize_tile<G>(a, x, base, (int64_t)blockIdx.x * Geom<G>::kGpc, tables_of(st), sj);
}

// Per-group parameters of the dequantizer: 2^z with z = log2(448 S) / k split
// as Pm 2^Pe, Pm = 2^(z - Pe) rounded once (in about [0.7, 1.42]) and Pe the
// integer nearest z, formed in double-float; 1/k as a double-float.  An
// all-zero group (S = 0) gets Pm = 0.
struct DequantGroup {
    float Pm;
    int Pe;
    float rk_hi, rk_lo;
    float P;   // Pm 2^Pe when that is a normal float, else 0 (the split path decides)
};

__device__ __forceinline__ DequantGroup dequant_group(float S, float k, const df::Tables& t) {
    DequantGroup d;
    const df::F2 rkd = df::recip21(k);
    d.rk_hi = rkd.hi;
    d.rk_lo = rkd.lo;
    if (!(S > 0.0f)) {
        d.Pm = 0.0f;
        d.Pe = 0;
        d.P = 0.0f;
        return d;
    }
    const df::F2 z = df::mul22(df::add2(df::log2_df(S, t), const_df(kLog2_448Df)), rkd);
    const float n0 = rintf(z.hi);
    d.Pm = df::exp2_df(df::F2{__fsub_rn(z.hi, n0), z.lo}, t);
    d.Pe = (int)n0;
    d.P = (d.Pe >= -125 && d.Pe <= 126) ? df::scale2(d.Pm, d.Pe) : 0.0f;
    return d;
}

// One code: sign(q) (|E4M3(q)| S)^(1/k) = sign(q) P 2^(L / k) with
// L = log2(|E4M3(q)| / 448) from the double-float table, |L / k| <= 17.8 / k.
// p = RN(L_hi / k) goes through the SFU exp2 (relative error <= 2^-22 for
// these arguments) and the rest of the double-float exponent, t (|t| <~ 2^-20),
// corrects it to first order: P (y + y t ln 2), y = 2^p.  The result is within
// about 2^-22 + 3 2^-24 of the exact value, 4.5e-7 (the codec's bar is 1e-6).
// When P is not a normal float (k < 1 with an extreme S) the group takes the
// split form: the integer part of the exponent applied exactly, the fraction
// through the SFU, a result outside the normal range scaled with one more
// rounding.
__device__ __forceinline__ float dequant_code(const float2* s_L, uint32_t code, const DequantGroup& d) {
    const uint32_t mag = code & 0x7Fu;
    if (mag == 0u || !(d.Pm > 0.0f)) return 0.0f;
    const float2 L = s_L[mag];
    const float p = __fmul_rn(L.x, d.rk_hi);
    const float t = fmaf(L.x, d.rk_lo, fmaf(L.y, d.rk_hi, fmaf(L.x, d.rk_hi, -p)));
    if (d.P > 0.0f) {
        const float y = ex2_ftz(p);
        const float x = __fmul_rn(d.P, fmaf(y, t * 0.693147182f, y));
        return __uint_as_float(__float_as_uint(x) | ((code & 0x80u) << 24));
    }
    const float rr = __fadd_rn(p, 12582912.0f);          // 1.5 2^23: rounds p to an integer
    const float n = __fsub_rn(rr, 12582912.0f);
    const float f = __fadd_rn(__fsub_rn(p, n), t);
    const float y = __fmul_rn(d.Pm, ex2_ftz(f));
    const int ni = (int)(__float_as_uint(rr) - 0x4B400000u) + d.Pe;
    const uint32_t yb = __float_as_uint(y);
    const int eb = (int)((yb >> 23) & 0xFFu) + ni;
    const float x = (eb >= 1 && eb <= 254) ? __uint_as_float(yb + ((uint32_t)ni << 23))
                                           : df::scale2(y, ni);
    return __uint_as_float(__float_as_uint(x) | ((code & 0x80u) << 24));
}

// The four codes of a packed word, all of one group whose P is a normal
// float: dequant_code's arithmetic two codes per packed f32x2 instruction
// (each half rounds like the scalar instruction, so the values are the same),
// -p formed directly as L (-1/k)_hi, zero magnitudes selected at the end.
__device__ __forceinline__ float4 dequant_word(const float2* s_L, uint32_t w, const DequantGroup& d) {
    const float2 L[4] = {s_L[w & 0x7Fu], s_L[(w >> 8) & 0x7Fu], s_L[(w >> 16) & 0x7Fu], s_L[(w >> 24) & 0x7Fu]};
    const uint64_t rh = pk(d.rk_hi, d.rk_hi), rl = pk(d.rk_lo, d.rk_lo), nrh = pk(-d.rk_hi, -d.rk_hi);
    const uint64_t ln2 = pk(0.693147182f, 0.693147182f), P = pk(d.P, d.P);
    float x[4];
#pragma unroll
    for (int h = 0; h < 4; h += 2) {
        const uint64_t lx = pk(L[h].x, L[h + 1].x), ly = pk(L[h].y, L[h + 1].y);
        const uint64_t np = mul2(lx, nrh);                                 // -p, exactly
        const uint64_t t = fma2(lx, rl, fma2(ly, rh, fma2(lx, rh, np)));
        float n0, n1;
        upk(np, n0, n1);
        const uint64_t y = pk(ex2_ftz(-n0), ex2_ftz(-n1));
        upk(mul2(P, fma2(y, mul2(t, ln2), y)), x[h], x[h + 1]);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t code = (w >> (8 * j)) & 0xFFu;
        x[j] = (code & 0x7Fu) ? __uint_as_float(__float_as_uint(x[j]) | ((code & 0x80u) << 24)) : 0.0f;
    }
    return make_float4(x[0], x[1], x[2], x[3]);
}

// Two 16-code chunks per thread (a CTA covers 2 x 4096 codes): the loads of
// both are issued before any arithmetic, so twice the bytes are in flight
// per thread (the per-code arithmetic is a dependent chain of ~15 operations).
constexpr int kDqChunks = 2;

template <int G>
__global__ void __launch_bounds__(kThreads)
dre_dequantize_kernel(const DequantArgs a) {
    using Gm = Geom<G>;
    constexpr int kCtaCodes = kDqChunks * kThreads * kVec;
    constexpr int kGpc = G >= 2 * kVec ? kCtaCodes / G : 1;   // groups per CTA (job form)
    __shared__ float2 s_L[128];
    __shared__ SmemTables st;
    __shared__ DequantGroup s_d[kGpc];
    const int64_t cta0 = (int64_t)blockIdx.x * kCtaCodes;
    // the codes first: their loads are in flight while the tables and groups are set up
    uint32_t q[kDqChunks][kVec / 4];
    int64_t base[kDqChunks];
    bool full[kDqChunks];
#pragma unroll
    for (int c = 0; c < kDqChunks; ++c) {
        base[c] = cta0 + (int64_t)(c * kThreads + threadIdx.x) * kVec;
        full[c] = base[c] + kVec <= a.n;
        if (full[c]) {
            const uint4 t = ld_cs(reinterpret_cast<const uint4*>(a.q + base[c]));
            q[c][0] = t.x; q[c][1] = t.y; q[c][2] = t.z; q[c][3] = t.w;
        } else {
#pragma unroll
            for (int i = 0; i < kVec / 4; ++i) q[c][i] = 0u;
#pragma unroll
            for (int e = 0; e < kVec; ++e)
                if (base[c] + e < a.n) q[c][e / 4] |= (uint32_t)a.q[base[c] + e] << (8 * (e & 3));
        }
    }
    for (int i = threadIdx.x; i < 128; i += kThreads)
        s_L[i] = make_float2(__uint_as_float(gtab::kLog2Frac448Hi[i]),
                             __uint_as_float(gtab::kLog2Frac448Lo[i]));
    load_smem_tables(st, threadIdx.x, kThreads);
    __syncthreads();
    const df::Tables tab = tables_of(st);
    if constexpr (Gm::kJobs) {
        // one thread per group of the CTA forms its dequantization parameters
        const int64_t gcta = cta0 / G;
        for (int j = threadIdx.x; j < kGpc; j += kThreads) {
            float S = 0.0f, k = 1.0f;
            if ((gcta + j) * G < a.n) { S = a.scale[gcta + j]; k = a.k[gcta + j]; }
            s_d[j] = dequant_group(S, k, tab);
        }
        __syncthreads();
    }
#pragma unroll
    for (int c = 0; c < kDqChunks; ++c) {
        if (base[c] >= a.n) continue;
        const int64_t g0 = base[c] / G;
        DequantGroup d[Gm::kGroups];
        if constexpr (Gm::kJobs) {
            d[0] = s_d[(int)(g0 - cta0 / G)];
        } else {
#pragma unroll
            for (int j = 0; j < Gm::kGroups; ++j) {
                float S = 0.0f, k = 1.0f;
                if ((g0 + j) * G < a.n) { S = a.scale[g0 + j]; k = a.k[g0 + j]; }
                d[j] = dequant_group(S, k, tab);
            }
        }
        float x[kVec];
#pragma unroll
        for (int i = 0; i < kVec / 4; ++i) {
            const DequantGroup& dw = d[(4 * i) / Gm::kElems];
            if (Gm::kElems >= 4 && dw.P > 0.0f) {   // the word's four codes share one group
                const float4 v = dequant_word(s_L, q[c][i], dw);
                x[4 * i] = v.x; x[4 * i + 1] = v.y; x[4 * i + 2] = v.z; x[4 * i + 3] = v.w;
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    x[4 * i + j] = dequant_code(s_L, (q[c][i] >> (8 * j)) & 0xFFu, d[(4 * i + j) / Gm::kElems]);
            }
        }
        if (full[c]) {
            float4* xp = reinterpret_cast<float4*>(a.x + base[c]);
#pragma unroll
            for (int i = 0; i < 4; ++i)
                st_cs(xp + i, make_float4(x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]));
        } else {
#pragma unroll
            for (int e = 0; e < kVec; ++e)
                if (base[c] + e < a.n) a.x[base[c] + e] = x[e];
        }
    }
}

// G >= 16: the CTA's 8192 codes as 64 rows of 128; warp w takes rows
// 8w .. 8w + 7 and each lane 4 consecutive codes of a row (one 32-bit load),
// so every warp store writes 512 contiguous bytes (the outputs are 4 of the 5
// bytes moved per code).  The groups' parameters are formed once per CTA, one
// thread per group, and shared.
constexpr int kDqRows = 64;
constexpr int kDqCtaCodes = kDqRows * 128;

template <int G>
__global__ void __launch_bounds__(kThreads)
dre_dequantize_rows_kernel(const DequantArgs a) {
    static_assert(G >= kVec, "row layout for G >= 16");
    constexpr int kGpc = kDqCtaCodes / G;   // groups per CTA
    constexpr int kRowsPerWarp = kDqRows / (kThreads / 32);
    __shared__ float2 s_L[128];
    __shared__ SmemTables st;
    __shared__ DequantGroup s_d[kGpc];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t cta0 = (int64_t)blockIdx.x * kDqCtaCodes;
    // the codes first: in flight while the tables and the groups are set up
    uint32_t q[kRowsPerWarp];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        const int64_t b = cta0 + (int64_t)(warp * kRowsPerWarp + r) * 128 + 4 * lane;
        if (b + 4 <= a.n) {
            q[r] = __ldcs(reinterpret_cast<const unsigned int*>(a.q + b));
        } else {
            q[r] = 0u;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (b + j < a.n) q[r] |= (uint32_t)a.q[b + j] << (8 * j);
        }
    }
    for (int i = threadIdx.x; i < 128; i += kThreads)
        s_L[i] = make_float2(__uint_as_float(gtab::kLog2Frac448Hi[i]),
                             __uint_as_float(gtab::kLog2Frac448Lo[i]));
    load_smem_tables(st, threadIdx.x, kThreads);
    __syncthreads();
    const df::Tables tab = tables_of(st);
    const int64_t gcta = cta0 / G;
    for (int j = threadIdx.x; j < kGpc; j += kThreads) {
        float S = 0.0f, k = 1.0f;
        if ((gcta + j) * G < a.n) { S = a.scale[gcta + j]; k = a.k[gcta + j]; }
        s_d[j] = dequant_group(S, k, tab);
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
        const int row = warp * kRowsPerWarp + r;
        const int64_t b = cta0 + (int64_t)row * 128 + 4 * lane;
        if (b >= a.n) break;
        const DequantGroup& d = s_d[(row * 128 + 4 * lane) / G];
        float x[4];
        if (d.P > 0.0f) {
            const float4 v = dequant_word(s_L, q[r], d);
            x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
        } else {   // an all-zero group, or P outside the normal range
#pragma unroll
            for (int j = 0; j < 4; ++j) x[j] = dequant_code(s_L, (q[r] >> (8 * j)) & 0xFFu, d);
        }
        if (b + 4 <= a.n) {
            st_cs(reinterpret_cast<float4*>(a.x + b), make_float4(x[0], x[1], x[2], x[3]));
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (b + j < a.n) a.x[b + j] = x[j];
        }
    }
}

// Plain per-group FP8 quantization without the expansion (section 3 FP8
// quantization equation alone: S = max|X| / 448, q = RNE(X / S), saturating):
// the reference point the expansion is measured against.
template <int G>
__global__ void __launch_bounds__(kThreads, G >= kVec ? 8 : 1)
absmax_quantize_kernel(const QuantArgs a) {
    using Gm = Geom<G>;
    const int64_t tid = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const int64_t base = tid * kVec;
    if (__all_sync(0xFFFFFFFFu, base >= a.n)) return;
    const bool active = base < a.n;
    const bool full = base + kVec <= a.n;

    float x[kVec];
    if (active && full) {
        const float4* xp = reinterpret_cast<const float4*>(a.x + base);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 t = ld_cs(xp + i);
            x[4 * i] = t.x; x[4 * i + 1] = t.y; x[4 * i + 2] = t.z; x[4 * i + 3] = t.w;
        }
    } else {
#pragma unroll
        for (int e = 0; e < kVec; ++e) x[e] = (active && base + e < a.n) ? a.x[base + e] : 0.0f;
    }
    float mx[Gm::kGroups];
#pragma unroll
    for (int j = 0; j < Gm::kGroups; ++j) mx[j] = 0.0f;
#pragma unroll
    for (int e = 0; e < kVec; ++e) mx[e / Gm::kElems] = fmaxf(mx[e / Gm::kElems], fabsf(x[e]));
#pragma unroll
    for (int off = Gm::kLanes / 2; off > 0; off >>= 1)
        mx[0] = fmaxf(mx[0], __shfl_xor_sync(0xFFFFFFFFu, mx[0], off));
    float S[Gm::kGroups], inv[Gm::kGroups];
#pragma unroll
    for (int j = 0; j < Gm::kGroups; ++j) {
        S[j] = __fdiv_rn(mx[j], 448.0f);
        inv[j] = rcp_approx(S[j]);
    }
    if (!active) return;

    uint32_t out[kVec / 4] = {0u, 0u, 0u, 0u}, und = 0u;
#pragma unroll
    for (int e = 0; e < kVec; ++e) {
        const int j = e / Gm::kElems;
        bool u;
        // an all-zero group keeps zero codes
        const uint32_t c = e4m3_code_fast(x[e], inv[j], u);
        if (S[j] > 0.0f) {
            out[e / 4] |= c << (8 * (e & 3));
            und |= (u ? 1u : 0u) << e;
        }
    }
    if (und) {   // rare: quotients beside a midpoint
#pragma unroll
        for (int e = 0; e < kVec; ++e) {
            if (und & (1u << e)) {
                const uint32_t c = e4m3_code_of_quotient_exact(x[e], S[e / Gm::kElems]);
                out[e / 4] = (out[e / 4] & ~(0xFFu << (8 * (e & 3)))) | (c << (8 * (e & 3)));
            }
        }
    }
#pragma unroll
    for (int i = 0; i < kVec / 4; ++i) out[i] = e4m3_canonical_zero(out[i]);
    if (full) {
        st_cs(reinterpret_cast<uint4*>(a.q + base), make_uint4(out[0], out[1], out[2], out[3]));
    } else {
#pragma unroll
        for (int e = 0; e < kVec; ++e)
            if (base + e < a.n) a.q[base + e] = (uint8_t)(out[e / 4] >> (8 * (e & 3)));
    }
    const int64_t g0 = base / G;
    const bool leader = G >= kVec ? ((base % G) == 0) : true;
    if (leader) {
#pragma unroll
        for (int j = 0; j < Gm::kGroups; ++j)
            if ((g0 + j) * G < a.n) a.scale[g0 + j] = S[j];
    }
}

template <int G>
cudaError_t launch_absmax(const QuantArgs& a, cudaStream_t s) {
    const int64_t threads = (a.n + kVec - 1) / kVec;
    absmax_quantize_kernel<G><<<(unsigned)((threads + kThreads - 1) / kThreads), kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

template <int G>
cudaError_t launch_q(const QuantArgs& a, cudaStream_t s) {
    const int64_t threads = (a.n + kVec - 1) / kVec;
    dre_quantize_kernel<G><<<(unsigned)((threads + kThreads - 1) / kThreads), kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

template <int G>
cudaError_t launch_dq(const DequantArgs& a, cudaStream_t s) {
    if constexpr (G >= kVec) {
        dre_dequantize_rows_kernel<G><<<(unsigned)((a.n + kDqCtaCodes - 1) / kDqCtaCodes), kThreads, 0, s>>>(a);
    } else {
        constexpr int64_t kCtaCodes = (int64_t)kDqChunks * kThreads * kVec;
        dre_dequantize_kernel<G><<<(unsigned)((a.n + kCtaCodes - 1) / kCtaCodes), kThreads, 0, s>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_absmax_quantize(const QuantArgs& a, int G, cudaStream_t s) {
    switch (G) {
        case 1: return launch_absmax<1>(a, s);
        case 2: return launch_absmax<2>(a, s);
        case 4: return launch_absmax<4>(a, s);
        case 8: return launch_absmax<8>(a, s);
        case 16: return launch_absmax<16>(a, s);
        case 32: return launch_absmax<32>(a, s);
        case 64: return launch_absmax<64>(a, s);
        case 128: return launch_absmax<128>(a, s);
        case 256: return launch_absmax<256>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_dre_quantize(const QuantArgs& a, int G, cudaStream_t s) {
    switch (G) {
        case 1: return launch_q<1>(a, s);
        case 2: return launch_q<2>(a, s);
        case 4: return launch_q<4>(a, s);
        case 8: return launch_q<8>(a, s);
        case 16: return launch_q<16>(a, s);
        case 32: return launch_q<32>(a, s);
        case 64: return launch_q<64>(a, s);
        case 128: return launch_q<128>(a, s);
        case 256: return launch_q<256>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_dre_dequantize(const DequantArgs& a, int G, cudaStream_t s) {
    switch (G) {
        case 1: return launch_dq<1>(a, s);
        case 2: return launch_dq<2>(a, s);
        case 4: return launch_dq<4>(a, s);
        case 8: return launch_dq<8>(a, s);
        case 16: return launch_dq<16>(a, s);
        case 32: return launch_dq<32>(a, s);
        case 64: return launch_dq<64>(a, s);
        case 128: return launch_dq<128>(a, s);
        case 256: return launch_dq<256>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace coat
