// act_quant.cu -- per-group (1 x G) FP8 quantization of an activation tensor
// with a transposed FP8 second output (COAT review page: section 3, Triton
// kernels, "non-linear layer optimisation": quantized FP8 output plus a
// transposed FP8 output for the backward pass; section 3, mixed-granularity
// activation quantization: 1 x G groups for non-linear layers; section 4
// table, group-scaling row: two-stage maximum reduction).
//
// x is an M x N bf16 tensor in row-major order.  Each row is split into
// groups of G consecutive elements; a group's scale is S = max|x| / 448 and its
// codes are E4M3(x / S), rounded to nearest even, saturating.  q holds the
// codes in the layout of x (M x N); qt holds the same codes transposed (N x M),
// so that the backward pass reads contiguous columns.
//
// A CTA owns a 64 x 128 tile: 128 threads quantize it row by row (8 elements
// per thread and pass, statistics per thread and then across the G/8 lanes of
// a group), store q and the scales, stage the codes in shared memory, and then
// write qt as 16-byte runs of one column, each built from 4 x 4 byte
// transposes.  The tile's inputs are copied into shared memory (cp.async) all
// at once when the CTA starts, so that its eight passes cost one memory
// latency without holding registers for the loads in flight.
#include <cstdint>

#include "coat_device.cuh"
#include "coat_kernels.h"

namespace coat {

namespace {

// RN(m / 448) for a bf16 group maximum m >= 0: q = RN(m y) with y = RN(1/448),
// then one FMA correction from the exact remainder m - q 448 (Markstein's
// division by a known divisor).  Checked against the correctly rounded
// quotient for every non-negative finite bf16 value, subnormals included.
constexpr float kInv448 = 1.0f / 448.0f;
__device__ __forceinline__ float div448_bf16(float m) {
    const float q = __fmul_rn(m, kInv448);
    const float r = fmaf(-q, 448.0f, m);
    return fmaf(r, kInv448, q);
}


// 16-byte asynchronous copy global -> shared (L2 only, no L1 allocation), and
// the wait for all of this thread's copies.
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    const uint32_t sa = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\ncp.async.wait_all;" ::: "memory");
}

constexpr int kTileR = 64;                  // rows per tile
constexpr int kTileC = 128;                 // columns per tile
constexpr int kActThreads = 128;
constexpr int kPitchW = kTileC / 4 + 1;     // shared-memory row pitch in words (padded)

template <int G>
__global__ void __launch_bounds__(kActThreads, 9)
act_quant_kernel(const ActArgs a) {
    __shared__ uint32_t tile[kTileR * kPitchW];
    __shared__ uint4 stage[kTileR / 8][kActThreads];   // the tile's inputs, [pass][thread]
    const int tid = threadIdx.x;
    const int64_t row0 = (int64_t)blockIdx.y * kTileR;
    const int64_t col0 = (int64_t)blockIdx.x * kTileC;
    const int64_t ngr = a.N / G;            // groups per row

    // ---- quantize: pass p covers rows 8p .. 8p+7, 16 threads per row ----
    const int r_in = tid >> 4;              // row within the pass
    const int c8 = (tid & 15) * 8;          // first column of this thread
    const bool col_ok = col0 + c8 < a.N;    // N % 16 == 0: all 8 columns or none
    // every pass's 16 bytes copied into shared memory at once (no registers
    // held while they are in flight); a thread reads back only its own slots,
    // so waiting for its own copies is enough
#pragma unroll
    for (int p = 0; p < kTileR / 8; ++p) {
        const int64_t rr = row0 + 8 * p + r_in;
        if (rr < a.M && col_ok) cp_async16(&stage[p][tid], a.x + rr * a.N + col0 + c8);
    }
    cp_async_wait_all();
#pragma unroll 1
    for (int p = 0; p < kTileR / 8; ++p) {
        const int64_t r = row0 + 8 * p + r_in;
        const uint4 v = (r < a.M && col_ok) ? stage[p][tid] : make_uint4(0u, 0u, 0u, 0u);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        float x[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[2 * i] = __uint_as_float(w[i] << 16);
            x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
        constexpr int kGroupsHere = G >= 8 ? 1 : 8 / G;   // groups in this thread's 8 elements
        constexpr int kPer = G >= 8 ? 8 : G;               // elements of one group here
        float S[kGroupsHere], inv[kGroupsHere];
        bool inv_bad = false;
#pragma unroll
        for (int j = 0; j < kGroupsHere; ++j) {
            float mx = 0.0f;
#pragma unroll
            for (int e = 0; e < kPer; e += 2) mx = max3(mx, fabsf(x[j * kPer + e]), fabsf(x[j * kPer + e + 1]));
            if constexpr (G > 8) {
#pragma unroll
                for (int off = G / 16; off > 0; off >>= 1)
                    mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
            }
            S[j] = div448_bf16(mx);
            // an all-zero group: inv = 0 keeps every code 0x00
            inv[j] = S[j] > 0.0f ? rcp_approx(S[j]) : 0.0f;
            inv_bad |= !(inv[j] <= 3.40282347e38f);
        }
        // codes of y (1 - 2^-20) and y (1 + 2^-20), two elements per conversion;
        // a byte that differs marks an element whose code a midpoint decides
        uint32_t codes[2] = {0u, 0u}, diff[2] = {0u, 0u};
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
            const uint64_t yy = fma2(pk(x[e], x[e + 1]), pk(inv[e / kPer], inv[(e + 1) / kPer]),
                                     pk(0.0f, 0.0f));   // +0 for a zero of either sign
            float l0, l1, h0, h1;
            upk(mul2(yy, pk(kDn, kDn)), l0, l1);
            upk(mul2(yy, pk(kUp, kUp)), h0, h1);
            const uint32_t clo = e4m3x2(l0, l1), chi = e4m3x2(h0, h1);
            codes[e / 4] |= clo << (16 * ((e >> 1) & 1));
            diff[e / 4] |= (clo ^ chi) << (16 * ((e >> 1) & 1));
        }
        if (inv_bad) {   // a subnormal scale: every element by division
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int sh = 8 * (e & 3);
                if (!(inv[e / kPer] <= 3.40282347e38f)) {
                    const uint32_t c = e4m3_code_of_quotient_exact(x[e], S[e / kPer]);
                    codes[e / 4] = (codes[e / 4] & ~(0xFFu << sh)) | (c << sh);
                    diff[e / 4] &= ~(0xFFu << sh);
                }
            }
        }
        if ((diff[0] | diff[1]) != 0u) {   // quotients beside a midpoint: the midpoint decides
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int wd = i >> 1, sh = 16 * (i & 1);
                const uint32_t d = (diff[wd] >> sh) & 0xFFFFu;
                if (d != 0u) {
                    const uint32_t lo = (codes[wd] >> sh) & 0xFFFFu;
                    const uint32_t c = e4m3x2_resolve(lo, lo ^ d, x[2 * i], x[2 * i + 1], S[(2 * i) / kPer],
                                                      S[(2 * i + 1) / kPer]);
                    codes[wd] = (codes[wd] & ~(0xFFFFu << sh)) | (c << sh);
                }
            }
        }
        codes[0] = e4m3_canonical_zero(codes[0]);
        codes[1] = e4m3_canonical_zero(codes[1]);
        const int tr = 8 * p + r_in;
        tile[tr * kPitchW + c8 / 4] = codes[0];
        tile[tr * kPitchW + c8 / 4 + 1] = codes[1];
        if (r < a.M && col_ok) {
            __stcs(reinterpret_cast<uint2*>(a.q + r * a.N + col0 + c8), make_uint2(codes[0], codes[1]));
            const int64_t g = (col0 + c8) / G;
            if constexpr (G >= 8) {
                if ((c8 % G) == 0) a.scale[r * ngr + g] = S[0];
            } else {
#pragma unroll
                for (int j = 0; j < kGroupsHere; ++j) a.scale[r * ngr + g + j] = S[j];
            }
        }
    }
    if (a.qt == nullptr) return;
    __syncthreads();

    // ---- transposed output: thread = (column quad, 16-row chunk) ----
    const int cq = tid & 31;                // columns 4 cq .. 4 cq + 3
    const int rc = tid >> 5;                // rows 16 rc .. 16 rc + 15
    const int64_t c_first = col0 + 4 * cq;
    const int64_t r_first = row0 + 16 * rc;
    if (c_first >= a.N || r_first >= a.M) return;   // N, M % 16 == 0: whole quads and chunks
    uint32_t col[4][4];                     // [column j][block b]: rows 4b .. 4b+3
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        const int tr = 16 * rc + 4 * b;
        const uint32_t w0 = tile[(tr + 0) * kPitchW + cq];
        const uint32_t w1 = tile[(tr + 1) * kPitchW + cq];
        const uint32_t w2 = tile[(tr + 2) * kPitchW + cq];
        const uint32_t w3 = tile[(tr + 3) * kPitchW + cq];
        const uint32_t t0 = __byte_perm(w0, w1, 0x5140);   // w0.b0 w1.b0 w0.b1 w1.b1
        const uint32_t t1 = __byte_perm(w2, w3, 0x5140);
        const uint32_t t2 = __byte_perm(w0, w1, 0x7362);   // w0.b2 w1.b2 w0.b3 w1.b3
        const uint32_t t3 = __byte_perm(w2, w3, 0x7362);
        col[0][b] = __byte_perm(t0, t1, 0x5410);
        col[1][b] = __byte_perm(t0, t1, 0x7632);
        col[2][b] = __byte_perm(t2, t3, 0x5410);
        col[3][b] = __byte_perm(t2, t3, 0x7632);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
        st_cs(reinterpret_cast<uint4*>(a.qt + (c_first + j) * a.M + r_first),
              make_uint4(col[j][0], col[j][1], col[j][2], col[j][3]));
}

template <int G>
cudaError_t launch_act(const ActArgs& a, cudaStream_t s) {
    const dim3 grid((unsigned)((a.N + kTileC - 1) / kTileC), (unsigned)((a.M + kTileR - 1) / kTileR));
    act_quant_kernel<G><<<grid, kActThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_act_quant(const ActArgs& a, int G, cudaStream_t s) {
    switch (G) {
        case 4: return launch_act<4>(a, s);
        case 8: return launch_act<8>(a, s);
        case 16: return launch_act<16>(a, s);
        case 32: return launch_act<32>(a, s);
        case 64: return launch_act<64>(a, s);
        case 128: return launch_act<128>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace coat
