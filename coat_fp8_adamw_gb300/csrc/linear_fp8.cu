// linear_fp8.cu -- FP8 linear layer with a per-group FP8 output (COAT review
// page: section 3, mixed-granularity activation quantization -- per-tensor FP8
// inputs for linear layers; section 3, Triton kernels, linear layer
// optimisation -- the output tile is reshaped to (BLOCK_M, BLOCK_N / G, G) and
// the maximum taken along the last axis, so the GEMM's epilogue emits the
// next layer's per-group FP8 activation directly).
//
//   y = (sx sw) (E4M3(xq) E4M3(wq)^T),  xq [M x K], wq [N x K] row-major codes
//   per row, groups of G consecutive columns:  S = RN(max|y| / 448),
//   q = E4M3(y / S) rounded to nearest even (of the exact quotient),
//   saturating, 0x00 for a quotient that rounds to zero (of either sign);
//   an all-zero group gets S = 0 and zero codes.
//
// The contraction runs on the tensor cores through the warp-level FP8 MMA
// (mma.sync m16n8k32, E4M3 x E4M3 -> fp32).  A CTA computes a 128 x 128
// output tile: its 8 warps own 16 rows each across all 128 columns, so every
// 1 x G group of a row lies in one warp and its maximum is a reduction over
// the 4 lanes of a quad (two shuffles).  K advances in steps of 64 through two
// shared-memory stages filled by cp.async; rows are padded to 80 bytes so
// that the 32-bit fragment loads of a warp hit 32 distinct banks.
#include <cstdint>

#include "coat_device.cuh"
#include "coat_kernels.h"

namespace coat {

namespace {

constexpr int kLBM = 128;                 // CTA tile rows (M)
constexpr int kLBN = 128;                 // CTA tile columns (N)
constexpr int kLBK = 64;                  // K per stage (bytes of a row)
constexpr int kLPitch = kLBK + 16;        // padded shared-memory row, bytes
constexpr int kLThreads = 256;            // 8 warps x 16 rows
constexpr int kLStage = kLBM * kLPitch;   // bytes of one operand stage

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// four 8 x 16-byte shared-memory matrices; lanes 8 i .. 8 i + 7 give the row
// addresses of matrix i, and lane l receives bytes 4 (l % 4) .. 4 (l % 4) + 3
// of row l / 4 of each (the m16n8k32 E4M3 fragment layout)
__device__ __forceinline__ void ldsm_x4(const unsigned char* p, uint32_t& r0, uint32_t& r1,
                                        uint32_t& r2, uint32_t& r3) {
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(p);
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(s));
}

// D += A B for a 16 x 32 E4M3 A (row-major fragment), a 32 x 8 E4M3 B
// (column-major fragment) and a 16 x 8 fp32 accumulator.
__device__ __forceinline__ void mma_e4m3(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// one stage: rows [0, 128) of A (from row m0) and of B (from row n0), bytes
// [k0, k0 + 64) of each row; 256 threads x 2 chunks of 16 bytes per operand
__device__ __forceinline__ void load_stage(const LinArgs& a, unsigned char* sA, unsigned char* sB,
                                           int64_t m0, int64_t n0, int64_t k0, int tid) {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const int c = tid + i * kLThreads;
        const int row = c >> 2, col = (c & 3) * 16;
        cp_async16(sA + row * kLPitch + col, a.xq + (m0 + row) * a.K + k0 + col);
        cp_async16(sB + row * kLPitch + col, a.wq + (n0 + row) * a.K + k0 + col);
    }
}

template <int G>
__global__ void __launch_bounds__(kLThreads, 2)
linear_fp8_kernel(const LinArgs a) {
    static_assert(G >= 8 && G <= kLBN && (kLBN % G) == 0, "G divides the tile");
    __shared__ __align__(16) unsigned char sA[2][kLStage];
    __shared__ __align__(16) unsigned char sB[2][kLStage];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gq = lane >> 2, tq = lane & 3;   // quad and lane within it
    const int64_t m0 = (int64_t)blockIdx.y * kLBM, n0 = (int64_t)blockIdx.x * kLBN;

    float acc[kLBN / 8][4];
#pragma unroll
    for (int j = 0; j < kLBN / 8; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.0f;

    const int64_t kt_n = a.K / kLBK;
    load_stage(a, sA[0], sB[0], m0, n0, 0, tid);
    cp_async_commit();
    for (int64_t kt = 0; kt < kt_n; ++kt) {
        const int s = (int)(kt & 1);
        if (kt + 1 < kt_n) load_stage(a, sA[s ^ 1], sB[s ^ 1], m0, n0, (kt + 1) * kLBK, tid);
        cp_async_commit();
        cp_async_wait<1>();   // this stage has landed (the next may be in flight)
        __syncthreads();
        // A fragment rows: lanes 0-7 rows 0-7 and 8-15 rows 8-15 at k, lanes
        // 16-31 the same rows at k + 16.  B: two n-blocks per ldmatrix, lanes
        // 0-7 / 8-15 the first block at k / k + 16, lanes 16-31 the second.
        const unsigned char* A = sA[s] + (warp * 16 + (lane & 15)) * kLPitch + (lane >> 4) * 16;
        const unsigned char* B = sB[s] + ((lane & 7) + (lane >> 4) * 8) * kLPitch + ((lane >> 3) & 1) * 16;
#pragma unroll
        for (int kk = 0; kk < kLBK; kk += 32) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4(A + kk, a0, a1, a2, a3);
#pragma unroll
            for (int j = 0; j < kLBN / 8; j += 2) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4(B + 8 * j * kLPitch + kk, b0, b1, b2, b3);
                mma_e4m3(acc[j], a0, a1, a2, a3, b0, b1);
                mma_e4m3(acc[j + 1], a0, a1, a2, a3, b2, b3);
            }
        }
        __syncthreads();   // the stage is free for the load two steps on
    }

    // ---- epilogue: scale, per-group maximum, scale and codes ----
    // This thread holds rows r0 and r0 + 8, columns 8 j + 2 tq + {0, 1}.
    const float sxw = __fmul_rn(a.sx, a.sw);
    const int64_t r0 = m0 + warp * 16 + gq;
    const int64_t ngr = a.N / G;   // groups per output row
    constexpr int kJ = G / 8;      // n-blocks per group
#pragma unroll
    for (int gi = 0; gi < kLBN / G; ++gi) {
        float y[2][2 * kJ];
        float mx0 = 0.0f, mx1 = 0.0f;
#pragma unroll
        for (int jj = 0; jj < kJ; ++jj) {
            const int j = gi * kJ + jj;
            y[0][2 * jj] = __fmul_rn(acc[j][0], sxw);
            y[0][2 * jj + 1] = __fmul_rn(acc[j][1], sxw);
            y[1][2 * jj] = __fmul_rn(acc[j][2], sxw);
            y[1][2 * jj + 1] = __fmul_rn(acc[j][3], sxw);
            mx0 = fmaxf(mx0, fmaxf(fabsf(y[0][2 * jj]), fabsf(y[0][2 * jj + 1])));
            mx1 = fmaxf(mx1, fmaxf(fabsf(y[1][2 * jj]), fabsf(y[1][2 * jj + 1])));
        }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, 2));
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t row = r0 + 8 * h;
            const float mx = h ? mx1 : mx0;
            const float S = __fdiv_rn(mx, 448.0f);
            const float inv = S > 0.0f ? rcp_approx(S) : 0.0f;
            const int64_t gcol = n0 / G + gi;
            if (tq == 0) a.scale[row * ngr + gcol] = S;
#pragma unroll
            for (int jj = 0; jj < kJ; ++jj) {
                const int64_t col = n0 + gi * G + 8 * jj + 2 * tq;
                uint32_t c2 = 0u;
                if (S > 0.0f) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        bool und;
                        uint32_t c = e4m3_code_fast(y[h][2 * jj + e], inv, und);
                        if (und) c = e4m3_code_of_quotient_exact(y[h][2 * jj + e], S);
                        c2 |= c << (8 * e);
                    }
                }
                *reinterpret_cast<uint16_t*>(a.q + row * a.N + col) = (uint16_t)e4m3_canonical_zero(c2);
                if (a.y)
                    *reinterpret_cast<float2*>(a.y + row * a.N + col) =
                        make_float2(y[h][2 * jj], y[h][2 * jj + 1]);
            }
        }
    }
}

template <int G>
cudaError_t launch_linear_g(const LinArgs& a, cudaStream_t s) {
    const dim3 grid((unsigned)(a.N / kLBN), (unsigned)(a.M / kLBM));
    linear_fp8_kernel<G><<<grid, kLThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_linear_fp8(const LinArgs& a, int G, cudaStream_t s) {
    switch (G) {
        case 8: return launch_linear_g<8>(a, s);
        case 16: return launch_linear_g<16>(a, s);
        case 32: return launch_linear_g<32>(a, s);
        case 64: return launch_linear_g<64>(a, s);
        case 128: return launch_linear_g<128>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace coat
