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
//   3. two-stage max / smallest-non-zero reduction of |m_t| and |v_t| per
//      group (stage 1 per thread over 16 elements, stage 2 warp shuffles
//      across the G/16 lanes of the group);
//   4. fresh k = log_{R_X}(R_E4M3) and S = max^k / 448 per group and moment;
//   5. re-expand, round to E4M3 and store codes, weights and (S, k).
//
// Layout: every thread owns 16 consecutive parameters, so each stream is
// whole 128-bit accesses: w 4x16 B, g 2x16 B, m codes 16 B, v codes 16 B;
// the 16-byte (S_m, k_m, S_v, k_v) record per group is one 128-bit access.
// A group of G >= 16 spans G/16 adjacent lanes of a warp; for G < 16 one
// thread holds 16/G whole groups.
#include "coat_kernels.h"
#include "coat_device.cuh"

namespace coat {

namespace {

template <int G>
struct Geom {
    static constexpr int kLanes = G >= kVec ? G / kVec : 1;          // lanes per group
    static constexpr int kGroups = G >= kVec ? 1 : kVec / G;         // groups per thread
    static constexpr int kElems = G >= kVec ? kVec : G;              // elements per (thread, group)
};

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
        // ragged tail: element-wise, absent elements read as zero
#pragma unroll
        for (int e = 0; e < kVec; ++e) {
            const bool in = base + e < a.n;
            c.w[e] = in ? a.w[base + e] : 0.0f;
            const uint32_t gb = in ? (uint32_t)a.g[base + e] : 0u;
            const uint32_t mb = in ? (uint32_t)a.mq[base + e] : 0u;
            const uint32_t vb = in ? (uint32_t)a.vq[base + e] : 0u;
            if ((e & 1) == 0) c.g[e / 2] = gb; else c.g[e / 2] |= gb << 16;
            if ((e & 3) == 0) { c.mq[e / 4] = mb; c.vq[e / 4] = vb; }
            else { c.mq[e / 4] |= mb << (8 * (e & 3)); c.vq[e / 4] |= vb << (8 * (e & 3)); }
        }
    }
}

template <int G>
__global__ void __launch_bounds__(kThreads)
adamw_dre_step_kernel(const StepArgs a) {
    using Gm = Geom<G>;
    __shared__ float s_log[128];
    if (threadIdx.x < 128) s_log[threadIdx.x] = __uint_as_float(kLog2Frac448Hi[threadIdx.x]);
    __syncthreads();

    const int64_t tid = (int64_t)blockIdx.x * kThreads + threadIdx.x;
    const int64_t base = tid * kVec;
    if (__all_sync(0xFFFFFFFFu, base >= a.n)) return;   // warp-uniform exit
    const bool active = base < a.n;
    const bool full = base + kVec <= a.n;

    Chunk c;
    if (active) load_chunk(a, base, full, c);
    else {
#pragma unroll
        for (int e = 0; e < kVec; ++e) c.w[e] = 0.0f;
#pragma unroll
        for (int i = 0; i < kVec / 2; ++i) c.g[i] = 0u;
#pragma unroll
        for (int i = 0; i < kVec / 4; ++i) { c.mq[i] = 0u; c.vq[i] = 0u; }
    }

    // per-group dequantization parameters of the stored state
    const int64_t g0 = base / G;   // first group touched by this thread
    DequantParams dm[Gm::kGroups], dv[Gm::kGroups];
#pragma unroll
    for (int j = 0; j < Gm::kGroups; ++j) {
        float4 md = make_float4(0.0f, 1.0f, 0.0f, 1.0f);
        if (active && (g0 + j) * G < a.n) md = ld_cs(a.meta + g0 + j);
        dm[j] = dequant_params(md.x, md.y);
        dv[j] = dequant_params(md.z, md.w);
    }

    // elementwise: dequantize, AdamW, stage-1 statistics
    float m[kVec], v[kVec];
    float mx_m[Gm::kGroups], mx_v[Gm::kGroups];
    uint32_t mn_m[Gm::kGroups], mn_v[Gm::kGroups];
#pragma unroll
    for (int j = 0; j < Gm::kGroups; ++j) {
        mx_m[j] = 0.0f; mx_v[j] = 0.0f; mn_m[j] = 0xFFFFFFFFu; mn_v[j] = 0xFFFFFFFFu;
    }
#pragma unroll
    for (int e = 0; e < kVec; ++e) {
        const int j = e / Gm::kElems;
        const uint32_t cm = (c.mq[e / 4] >> (8 * (e & 3))) & 0xFFu;
        const uint32_t cv = (c.vq[e / 4] >> (8 * (e & 3))) & 0xFFu;
        const float m_prev = dequant_one(s_log, cm, dm[j].P, dm[j].rk);
        const float v_prev = dequant_one(s_log, cv, dv[j].P, dv[j].rk);
        const float gf = (e & 1) ? bf16_hi(c.g[e / 2]) : bf16_lo(c.g[e / 2]);
        const float mt = fmaf(a.beta1, m_prev, __fmul_rn(a.omb1, gf));
        const float vt = fmaf(a.beta2, v_prev, __fmul_rn(__fmul_rn(a.omb2, gf), gf));
        const float denom = __fadd_rn(sqrt_approx(__fmul_rn(vt, a.c2)), a.eps);
        c.w[e] = fmaf(__fmul_rn(-a.c1, mt), rcp_approx(denom), __fmul_rn(c.w[e], a.decay));
        m[e] = mt;
        v[e] = vt;
        const float am = fabsf(mt);
        mx_m[j] = fmaxf(mx_m[j], am);
        mx_v[j] = fmaxf(mx_v[j], vt);
        mn_m[j] = min(mn_m[j], nz_key(am));
        mn_v[j] = min(mn_v[j], nz_key(vt));
    }

    // stage 2: across the lanes of a group
#pragma unroll
    for (int off = Gm::kLanes / 2; off > 0; off >>= 1) {
        mx_m[0] = fmaxf(mx_m[0], __shfl_xor_sync(0xFFFFFFFFu, mx_m[0], off));
        mx_v[0] = fmaxf(mx_v[0], __shfl_xor_sync(0xFFFFFFFFu, mx_v[0], off));
        mn_m[0] = min(mn_m[0], __shfl_xor_sync(0xFFFFFFFFu, mn_m[0], off));
        mn_v[0] = min(mn_v[0], __shfl_xor_sync(0xFFFFFFFFu, mn_v[0], off));
    }

    // fresh (k, S) per group and moment
    QuantParams qm[Gm::kGroups], qv[Gm::kGroups];
#pragma unroll
    for (int j = 0; j < Gm::kGroups; ++j) {
        qm[j] = quant_params(mx_m[j], nz_key_value(mn_m[j]));
        qv[j] = quant_params(mx_v[j], nz_key_value(mn_v[j]));
    }
    if (!active) return;

    // an fp32-subnormal group max has no finite reciprocal: pre-scale by 2^24
    bool tiny = false;
#pragma unroll
    for (int j = 0; j < Gm::kGroups; ++j) tiny |= (mx_m[j] < 1.17549435e-38f) | (mx_v[j] < 1.17549435e-38f);
    float pre_m[Gm::kGroups], pre_v[Gm::kGroups];
#pragma unroll
    for (int j = 0; j < Gm::kGroups; ++j) {
        pre_m[j] = 1.0f;
        pre_v[j] = 1.0f;
        if (tiny) {
            if (mx_m[j] < 1.17549435e-38f && mx_m[j] > 0.0f) { pre_m[j] = 16777216.0f; qm[j].inv_mx = __frcp_rn(mx_m[j] * 16777216.0f); }
            if (mx_v[j] < 1.17549435e-38f && mx_v[j] > 0.0f) { pre_v[j] = 16777216.0f; qv[j].inv_mx = __frcp_rn(mx_v[j] * 16777216.0f); }
        }
    }

    // re-expand and encode
    uint32_t om[kVec / 4], ov[kVec / 4];
#pragma unroll
    for (int e = 0; e < kVec; e += 2) {
        const int j = e / Gm::kElems;
        const int j1 = (e + 1) / Gm::kElems;
        float r0m = fabsf(m[e]) * qm[j].inv_mx, r1m = fabsf(m[e + 1]) * qm[j1].inv_mx;
        float r0v = v[e] * qv[j].inv_mx, r1v = v[e + 1] * qv[j1].inv_mx;
        if (tiny) {
            r0m = (fabsf(m[e]) * pre_m[j]) * qm[j].inv_mx;
            r1m = (fabsf(m[e + 1]) * pre_m[j1]) * qm[j1].inv_mx;
            r0v = (v[e] * pre_v[j]) * qv[j].inv_mx;
            r1v = (v[e + 1] * pre_v[j1]) * qv[j1].inv_mx;
        }
        const uint32_t pm = e4m3x2(expand_scaled(m[e], r0m, qm[j].k), expand_scaled(m[e + 1], r1m, qm[j1].k));
        const uint32_t pv = e4m3x2(expand_scaled(v[e], r0v, qv[j].k), expand_scaled(v[e + 1], r1v, qv[j1].k));
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
    // one lane per group writes the group record
    const bool leader = G >= kVec ? ((base % G) == 0) : true;
    if (leader) {
#pragma unroll
        for (int j = 0; j < Gm::kGroups; ++j)
            if ((g0 + j) * G < a.n)
                st_cs(a.meta + g0 + j, make_float4(qm[j].S, qm[j].k, qv[j].S, qv[j].k));
    }
}

template <int G>
cudaError_t launch_step(const StepArgs& a, cudaStream_t stream) {
    const int64_t threads = (a.n + kVec - 1) / kVec;
    const int64_t blocks = (threads + kThreads - 1) / kThreads;
    adamw_dre_step_kernel<G><<<(unsigned)blocks, kThreads, 0, stream>>>(a);
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
