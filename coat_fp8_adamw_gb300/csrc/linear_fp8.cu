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
// Blackwell organisation: persistent CTA pairs (clusters of two, one CTA per
// SM) walk the 256 x 256 output tiles.  Each CTA streams its 128 rows of X and
// its 128 rows of W (half the tile's columns) in 128-byte K slices into a
// 6-stage shared-memory ring with TMA (128-byte swizzle), both signalling the
// even CTA's barrier.  One thread of the even CTA issues the pair-wide
// fifth-generation tensor-core MMA (tcgen05.mma.cta_group::2 kind::f8f6f4,
// M = 256, N = 256, K = 32, E4M3 x E4M3 -> f32): each SM multiplies its own
// 128 rows of X by both halves of W, so a CTA loads a third less per FLOP than
// a single-SM 128 x 256 tile.  Accumulators alternate between two 256-column
// halves of tensor memory; eight epilogue warps per CTA (two per SM
// sub-partition, each taking 128 of the 256 columns) read their CTA's 128
// rows back (tcgen05.ld, one output row per thread, so a 1 x G group lies in
// one thread's registers) and run the scale-and-quantize epilogue while the
// next tile accumulates.  Every wait on an mbarrier is bounded: when one gives up,
// the kernel counts it in g_wait_timeouts, lets its copies and MMAs in flight
// finish, frees its tensor memory and returns.
#include <atomic>
#include <cstdint>
#include <cuda.h>   // CUtensorMap and its enums; the encoder is fetched at run time

#include "coat_device.cuh"
#include "coat_kernels.h"

namespace coat {

__device__ unsigned long long g_wait_timeouts;

namespace {

constexpr int kBM = 128;                       // rows of X per CTA (the pair's MMA has M = 256)
constexpr int kBN = 256;                       // tile columns (N) = the MMA's N
constexpr int kBNh = kBN / 2;                  // rows of W per CTA
constexpr int kBK = 128;                       // K bytes per stage: one 128-byte swizzle row
constexpr int kMmaK = 32;                      // K of one kind::f8f6f4 MMA
constexpr int kStages = 6;
constexpr int kABytes = kBM * kBK;             // 16 KB
constexpr int kBBytes = kBNh * kBK;            // 16 KB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kEpiWarps = 8;                   // two per SM sub-partition, each half the columns
constexpr int kEpiCols = kBN / (kEpiWarps / 4);
constexpr int kThreads = 32 * (4 + kEpiWarps);
constexpr uint32_t kTmemCols = 2 * kBN;        // two accumulators of 256 f32 columns
constexpr int kBarOff = kStages * kStageBytes;
constexpr int kNumBars = 2 * kStages + 5;      // full, empty, acc full x2, acc empty x2, done
constexpr int kSmemBytes = kBarOff + 8 * kNumBars + 16 + 1024;   // + slack for 1024-B alignment
constexpr uint32_t kSpinLimit = 1u << 26;

// Instruction descriptor of the pair's MMA: D in f32 (bits 4-5 = 1), A and B
// E4M3 (bits 7-9 and 10-12 = 0), both K-major (bits 15, 16 = 0), N / 8 in
// bits 17-22, M / 16 in bits 24-28 (M = 256 over the two CTAs).
constexpr uint32_t kIdesc = (1u << 4) | ((uint32_t)(kBN >> 3) << 17) | ((uint32_t)((2 * kBM) >> 4) << 24);

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

// ---- mbarriers ----
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0u;
}
// Wait for the phase of parity `parity` to complete, at most kSpinLimit
// polls; give up early once another role has aborted (when `abort` is given).
__device__ __noinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile uint32_t* abort) {
    for (uint32_t i = 0; i < kSpinLimit; ++i) {
        if (mbar_try(bar, parity)) return true;
        if (abort && (i & 255u) == 255u && *abort) return false;
    }
    atomicAdd(&g_wait_timeouts, 1ull);
    if (abort) *abort = 1u;
    return false;
}
// the common case (the phase has already completed) without the call
__device__ __forceinline__ bool mbar_wait_fast(uint32_t bar, uint32_t parity, volatile uint32_t* abort) {
    return mbar_try(bar, parity) || mbar_wait(bar, parity, abort);
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// arrive on an mbarrier of either CTA of the cluster (a shared::cluster address)
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cbar) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cbar) : "memory");
}

// ---- clusters ----
__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// the shared::cluster address of this CTA's shared address `a` in CTA `rank`
__device__ __forceinline__ uint32_t map_to_rank(uint32_t a, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
    return r;
}
// every thread of both CTAs (the non-.aligned form: lanes of a warp may arrive apart)
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

// ---- TMA ----
// A 2-D tile into this CTA's shared memory, its bytes counted on `cbar`, an
// mbarrier of either CTA of the pair (shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, int32_t x, int32_t y,
                                                 uint32_t cbar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2 "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(cbar)
        : "memory");
}

// ---- tcgen05 ----
// Shared-memory matrix descriptor of a K-major operand in the 128-byte
// swizzled layout TMA writes: rows of 128 bytes, 8-row (1024-byte) swizzle
// atoms.  Start address / 16 in bits 0-13, leading-dimension offset (unused
// by this layout) in bits 16-29, stride between 8-row atoms / 16 in bits
// 32-45, the descriptor version 1 in bits 46-47, swizzle mode 2 (128 bytes)
// in bits 61-63.  A K offset inside the 128-byte row is added to the start
// address: the swizzle is a function of the address bits.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
__device__ __forceinline__ void mma_e4m3_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                              uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(kIdesc), "r"(accumulate)
        : "memory");
}
// arrive on the mbarrier at shared address `bar` in every CTA of `mask` once
// every MMA this thread issued before has completed
__device__ __forceinline__ void mma_commit_pair(uint32_t bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
        "h"(mask)
        : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 lanes x N consecutive 32-bit columns: thread i receives lane (taddr's lane + i)
// (the wait for the registers is part of the same statement)
template <int N>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, uint32_t (&r)[N]);
template <>
__device__ __forceinline__ void tmem_ld<32>(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
        "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
        "%30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
          "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
          "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
          "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// Codes of 2 n values of one row, y = RN(acc sxw), on the packed f32x2 path:
// the codes of y inv (1 -+ 2^-20) agree when no E4M3 midpoint lies near
// y / S, and the rare elements where they differ (or where the reciprocal is
// not finite) are decided from the exact quotient.  inv[e / kPer] and
// S[e / kPer] belong to element e.
template <int n, int kPer>
__device__ __forceinline__ void codes_of(const uint32_t* v, float sxw, const float* S, const float* inv,
                                         float* y, uint32_t* w) {
    const uint64_t sxw2 = pk(sxw, sxw), zero2 = pk(0.0f, 0.0f), dn2 = pk(kDn, kDn), up2 = pk(kUp, kUp);
    uint32_t dw[n / 4];
#pragma unroll
    for (int e = 0; e < n; e += 2) {
        const uint64_t y2 = mul2(pk(__uint_as_float(v[e]), __uint_as_float(v[e + 1])), sxw2);
        upk(y2, y[e], y[e + 1]);
        const uint64_t yy = fma2(y2, pk(inv[e / kPer], inv[(e + 1) / kPer]), zero2);   // +0 for -0
        float l0, l1, h0, h1;
        upk(mul2(yy, dn2), l0, l1);
        upk(mul2(yy, up2), h0, h1);
        const uint32_t clo = e4m3x2(l0, l1), chi = e4m3x2(h0, h1);
        if ((e & 2) == 0) { w[e / 4] = clo; dw[e / 4] = clo ^ chi; }
        else { w[e / 4] |= clo << 16; dw[e / 4] |= (clo ^ chi) << 16; }
    }
    uint32_t any = 0u;
#pragma unroll
    for (int i = 0; i < n / 4; ++i) any |= dw[i];
#pragma unroll
    for (int j = 0; j < (n + kPer - 1) / kPer; ++j) any |= (inv[j] <= 3.40282347e38f) ? 0u : 1u;
    if (any != 0u) {   // rare: quotients beside a midpoint
#pragma unroll
        for (int e = 0; e < n; ++e) {
            const int sh = 8 * (e & 3);
            const bool bad = !(inv[e / kPer] <= 3.40282347e38f);
            if (S[e / kPer] > 0.0f && (bad || ((dw[e / 4] >> sh) & 0xFFu) != 0u)) {
                const uint32_t code = e4m3_code_of_quotient_exact(y[e], S[e / kPer]);
                w[e / 4] = (w[e / 4] & ~(0xFFu << sh)) | (code << sh);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < n / 4; ++i) w[i] = e4m3_canonical_zero(w[i]);
}

// the codes (and y when asked for) of n columns from col of this thread's row
template <int n>
__device__ __forceinline__ void store_codes(const LinArgs& a, int64_t row, int64_t col, const uint32_t* w,
                                            const float* y) {
    uint8_t* qp = a.q + row * a.N + col;
    if constexpr (n == 8) {
        *reinterpret_cast<uint2*>(qp) = make_uint2(w[0], w[1]);
    } else {
#pragma unroll
        for (int i = 0; i < n / 16; ++i)
            reinterpret_cast<uint4*>(qp)[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
    }
    if (a.y) {
        float4* yp = reinterpret_cast<float4*>(a.y + row * a.N + col);
#pragma unroll
        for (int i = 0; i < n / 4; ++i) yp[i] = make_float4(y[4 * i], y[4 * i + 1], y[4 * i + 2], y[4 * i + 3]);
    }
}

// One tile's epilogue for this thread: one output row, kEpiCols columns from
// n0.  Per group of G columns: max|acc| (|RN(acc sxw)| is monotone in |acc|,
// so max|y| = RN(max|acc| sxw)), S = RN(max|y| / 448), then the codes.
// Columns come from tensor memory 32 at a time: a chunk holds 32 / G whole
// groups when G <= 32, and a wider group is read twice (maximum, then codes)
// instead of being held in registers.
template <int G>
__device__ __forceinline__ void epilogue_row(const LinArgs& a, uint32_t taddr, int64_t row, int64_t n0,
                                             float sxw) {
    constexpr int kCh = 32;
    const bool row_ok = row < a.M;
    const int64_t ngr = a.N / G;
    if constexpr (G <= kCh) {
        constexpr int kGpc = kCh / G;
#pragma unroll 1
        for (int c = 0; c < kEpiCols / kCh; ++c) {
            const int64_t col0 = n0 + (int64_t)c * kCh;
            if (col0 >= a.N) break;   // the same for the whole warp
            uint32_t v[kCh];
            __syncwarp();   // tcgen05.ld is warp-collective: converge after the code branches
            tmem_ld<kCh>(taddr + (uint32_t)(c * kCh), v);
            float S[kGpc], inv[kGpc];
#pragma unroll
            for (int j = 0; j < kGpc; ++j) {
                float mxa = 0.0f;
#pragma unroll
                for (int e = j * G; e < (j + 1) * G; e += 2)
                    mxa = max3(mxa, fabsf(__uint_as_float(v[e])), fabsf(__uint_as_float(v[e + 1])));
                S[j] = __fdiv_rn(__fmul_rn(mxa, sxw), 448.0f);
                inv[j] = S[j] > 0.0f ? rcp_approx(S[j]) : 0.0f;
            }
            float y[kCh];
            uint32_t w[kCh / 4];
            codes_of<kCh, G>(v, sxw, S, inv, y, w);
            if (row_ok) {
                const int64_t si = row * ngr + col0 / G;
                if (col0 + kCh <= a.N) {   // the whole chunk: one store of codes, scales together
                    store_codes<kCh>(a, row, col0, w, y);
                    if constexpr (kGpc == 4) {
                        if ((si & 3) == 0) *reinterpret_cast<float4*>(a.scale + si) = make_float4(S[0], S[1], S[2], S[3]);
                        else for (int j = 0; j < 4; ++j) a.scale[si + j] = S[j];
                    } else if constexpr (kGpc == 2) {
                        if ((si & 1) == 0) *reinterpret_cast<float2*>(a.scale + si) = make_float2(S[0], S[1]);
                        else for (int j = 0; j < 2; ++j) a.scale[si + j] = S[j];
                    } else {
                        a.scale[si] = S[0];
                    }
                } else {   // N is a multiple of G, not of the chunk
#pragma unroll
                    for (int j = 0; j < kGpc; ++j) {
                        const int64_t col = col0 + j * G;
                        if (col < a.N) {
                            a.scale[si + j] = S[j];
                            store_codes<G>(a, row, col, w + j * (G / 4), y + j * G);
                        }
                    }
                }
            }
        }
    } else {
        constexpr int kNch = G / kCh;
#pragma unroll 1
        for (int g = 0; g < kEpiCols / G; ++g) {
            const int64_t col0 = n0 + (int64_t)g * G;
            if (col0 >= a.N) break;
            uint32_t v[kCh];
            float mxa = 0.0f;
#pragma unroll
            for (int c = 0; c < kNch; ++c) {
                __syncwarp();
                tmem_ld<kCh>(taddr + (uint32_t)(g * G + c * kCh), v);
#pragma unroll
                for (int e = 0; e < kCh; e += 2)
                    mxa = max3(mxa, fabsf(__uint_as_float(v[e])), fabsf(__uint_as_float(v[e + 1])));
            }
            const float S = __fdiv_rn(__fmul_rn(mxa, sxw), 448.0f);
            const float inv = S > 0.0f ? rcp_approx(S) : 0.0f;
            if (row_ok) a.scale[row * ngr + col0 / G] = S;
#pragma unroll
            for (int c = 0; c < kNch; ++c) {
                __syncwarp();
                tmem_ld<kCh>(taddr + (uint32_t)(g * G + c * kCh), v);
                float y[kCh];
                uint32_t w[kCh / 4];
                codes_of<kCh, kCh>(v, sxw, &S, &inv, y, w);
                if (row_ok) store_codes<kCh>(a, row, col0 + c * kCh, w, y);
            }
        }
    }
}

// Tile order: bands of kGroupM row pairs, column-major inside a band, so the
// pairs running at once share a band of X (kGroupM x 256 rows, kept in L2)
// and walk W together, instead of all sweeping X for every column block.
constexpr int64_t kGroupM = 16;
struct TileCoord {
    int64_t m, n;   // row-pair block (256 rows) and column block (256 columns)
};
__device__ __forceinline__ TileCoord tile_coord(int64_t t, int64_t num_m, int64_t num_n) {
    const int64_t band = t / (kGroupM * num_n), first = band * kGroupM;
    const int64_t rows = num_m - first < kGroupM ? num_m - first : kGroupM;
    const int64_t r = t - band * kGroupM * num_n;
    return TileCoord{first + r % rows, r / rows};
}

template <int G>
__global__ void __launch_bounds__(kThreads, 1)
linear_fp8_kernel(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmw,
                  const LinArgs a) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // the 128-byte swizzle repeats every 1024 bytes: align the stages to it
    // (the same offset in both CTAs of the pair: the MMA addresses both rings
    // with one descriptor)
    const uint32_t raw = smem_u32(smem_raw);
    unsigned char* smem = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    const uint32_t sb = smem_u32(smem);
    const uint32_t bar0 = sb + kBarOff;
    auto full = [&](int s) { return bar0 + 8u * (uint32_t)s; };
    auto empty = [&](int s) { return bar0 + 8u * (uint32_t)(kStages + s); };
    auto acc_full = [&](int b) { return bar0 + 8u * (uint32_t)(2 * kStages + b); };
    auto acc_empty = [&](int b) { return bar0 + 8u * (uint32_t)(2 * kStages + 2 + b); };
    const uint32_t done = bar0 + 8u * (uint32_t)(2 * kStages + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kBarOff + 8 * kNumBars);
    volatile uint32_t* abort = tmem_slot + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();   // 0: the CTA that issues the pair's MMAs
    const bool leader = rank == 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) { mbar_init(full(s), 1); mbar_init(empty(s), 1); }
        // the leader's accumulator is free once every epilogue warp of both CTAs is done with it
        for (int b = 0; b < 2; ++b) { mbar_init(acc_full(b), 1); mbar_init(acc_empty(b), 2 * kEpiWarps); }
        mbar_init(done, 1);
        *abort = 0u;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmx)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmw)) : "memory");
    }
    if (warp == 2) {
        // the same columns in both CTAs of the pair
        asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    cluster_sync();   // barriers initialised and tensor memory allocated in both CTAs
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const int64_t num_m = (a.M + 2 * kBM - 1) / (2 * kBM), num_n = (a.N + kBN - 1) / kBN;
    const int64_t tiles = num_m * num_n;
    const int kblocks = (int)((a.K + kBK - 1) / kBK);
    const int64_t cid = blockIdx.x >> 1, nclusters = gridDim.x >> 1;

    if (warp == 0 && lane == 0) {
        // ---- TMA producer (both CTAs): this CTA's rows of X and of W ----
        int s = 0;
        uint32_t ph = 0, issued = 0, last_ph = 0;   // per stage: issued at all, parity of the last issue
        bool ok = true;
        const uint32_t fb0 = map_to_rank(full(0), 0);   // the leader's barriers, contiguous like ours
        for (int64_t t = cid; ok && t < tiles; t += nclusters) {
            const TileCoord tc = tile_coord(t, num_m, num_n);
            const int32_t m0 = (int32_t)(tc.m * (2 * kBM) + rank * kBM);
            const int32_t n0 = (int32_t)(tc.n * kBN + rank * kBNh);
            for (int kb = 0; kb < kblocks; ++kb) {
                if (!mbar_wait_fast(empty(s), ph ^ 1u, abort)) { ok = false; break; }
                // the leader's barrier counts the bytes of both CTAs
                if (leader) mbar_expect_tx(full(s), (uint32_t)(2 * kStageBytes));
                const uint32_t fb = fb0 + 8u * (uint32_t)s;
                const uint32_t sa = sb + (uint32_t)(s * kStageBytes);
                tma_load_2d_pair(sa, &tmx, kb * kBK, m0, fb);
                tma_load_2d_pair(sa + kABytes, &tmw, kb * kBK, n0, fb);
                issued |= 1u << s;
                last_ph = (last_ph & ~(1u << s)) | (ph << s);
                if (++s == kStages) { s = 0; ph ^= 1u; }
            }
        }
        // every stage issued has been read by the MMAs (and the release that
        // says so has landed here) before the CTA may exit
        for (int i = 0; i < kStages; ++i)
            if (issued & (1u << i)) mbar_wait(empty(i), (last_ph >> i) & 1u, nullptr);
    } else if (warp == 1 && lane == 0) {
        if (leader) {
            // ---- MMA issuer (even CTA) ----
            int s = 0, acc = 0;
            uint32_t ph = 0, aph = 0;
            bool ok = true;
            // descriptors of stage 0; a stage / K step moves only the start
            // address field (address / 16, 14 bits, no carry out for shared addresses)
            const uint64_t adesc0 = sw128_desc(sb), bdesc0 = sw128_desc(sb + kABytes);
            for (int64_t t = cid; ok && t < tiles; t += nclusters) {
                if (!mbar_wait_fast(acc_empty(acc), aph ^ 1u, abort)) break;
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(acc * kBN);
                for (int kb = 0; kb < kblocks; ++kb) {
                    if (!mbar_wait_fast(full(s), ph, abort)) { ok = false; break; }
                    tc_fence_after();
                    const uint64_t so = (uint64_t)(s * (kStageBytes >> 4));
#pragma unroll
                    for (int kk = 0; kk < kBK / kMmaK; ++kk)
                        mma_e4m3_pair(d, adesc0 + so + (uint64_t)(kk * (kMmaK >> 4)),
                                      bdesc0 + so + (uint64_t)(kk * (kMmaK >> 4)), (kb | kk) != 0);
                    mma_commit_pair(empty(s), 0x3);   // both CTAs' stage s is free once read
                    if (++s == kStages) { s = 0; ph ^= 1u; }
                }
                if (!ok) break;
                mma_commit_pair(acc_full(acc), 0x3);
                acc ^= 1;
                if (acc == 0) aph ^= 1u;
            }
            // every MMA issued has completed before either CTA frees tensor memory
            mma_commit_pair(done, 0x3);
        }
        mbar_wait(done, 0u, nullptr);
    } else if (warp >= 4) {
        // ---- epilogue: warp w reads tensor-memory lanes 32 (w % 4) .. 32 (w % 4) + 31
        // (the sub-partition it runs on), columns kEpiCols (w - 4) / 4 onwards ----
        const int q4 = warp & 3, ch = (warp - 4) >> 2;
        const float sxw = __fmul_rn(a.sx, a.sw);
        int acc = 0;
        uint32_t aph = 0;
        for (int64_t t = cid; t < tiles; t += nclusters) {
            if (!mbar_wait_fast(acc_full(acc), aph, abort)) break;
            tc_fence_after();
            const TileCoord tc = tile_coord(t, num_m, num_n);
            const int64_t row = tc.m * (2 * kBM) + rank * kBM + 32 * q4 + lane;
            const uint32_t taddr = tmem + ((uint32_t)(32 * q4) << 16) + (uint32_t)(acc * kBN + ch * kEpiCols);
            epilogue_row<G>(a, taddr, row, tc.n * kBN + ch * kEpiCols, sxw);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(map_to_rank(acc_empty(acc), 0));
            acc ^= 1;
            if (acc == 0) aph ^= 1u;
        }
    }
    tc_fence_before();
    cluster_sync();   // no arrival or copy is still on its way to either CTA
    tc_fence_after();
    if (warp == 2)
        asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                     : "memory");
}

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                 CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                 CUtensorMapFloatOOBfill);

EncodeTiled encoder() {
    static const EncodeTiled fn = []() -> EncodeTiled {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<EncodeTiled>(p);
    }();
    return fn;
}

// rows x K bytes, row-major; boxes of 128 bytes x box_rows rows, 128-byte swizzle,
// zeros outside the tensor
bool encode_operand(CUtensorMap* map, const uint8_t* base, int64_t rows, int64_t K, uint32_t box_rows) {
    const EncodeTiled fn = encoder();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)K};
    const cuuint32_t box[2] = {(cuuint32_t)kBK, box_rows};
    const cuuint32_t elem[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(base), dims, strides, box, elem,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Per device and G: the number of CTA pairs that fit at once, a property of
// the device and the kernel (0 = not known yet; set once, read without a lock:
// a race only repeats the same host-side query).  The shared-memory attribute
// is set on every launch, since a device reset clears it.
constexpr int kMaxDevices = 64;
std::atomic<int> g_pairs[kMaxDevices][5];

int g_index(int G) { return G == 8 ? 0 : G == 16 ? 1 : G == 32 ? 2 : G == 64 ? 3 : 4; }

template <int G>
cudaError_t launch_linear_g(const LinArgs& a, cudaStream_t s) {
    alignas(64) CUtensorMap tmx, tmw;
    if (!encode_operand(&tmx, a.xq, a.M, a.K, kBM) || !encode_operand(&tmw, a.wq, a.N, a.K, kBNh))
        return cudaErrorInvalidValue;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::atomic<int>* cached = (dev >= 0 && dev < kMaxDevices) ? &g_pairs[dev][g_index(G)] : nullptr;
    int clusters = cached ? cached->load(std::memory_order_relaxed) : 0;
    e = cudaFuncSetAttribute(linear_fp8_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3(2);
    if (clusters < 1) {   // first launch on this device
        if ((e = cudaOccupancyMaxActiveClusters(&clusters, linear_fp8_kernel<G>, &cfg)) != cudaSuccess) return e;
        if (clusters < 1) return cudaErrorInvalidConfiguration;
        if (cached) cached->store(clusters, std::memory_order_relaxed);
    }
    const int64_t tiles = ((a.M + 2 * kBM - 1) / (2 * kBM)) * ((a.N + kBN - 1) / kBN);
    cfg.gridDim = dim3(2u * (unsigned)(tiles < clusters ? tiles : clusters));
    e = cudaLaunchKernelEx(&cfg, linear_fp8_kernel<G>, tmx, tmw, a);
    if (e != cudaSuccess) return e;
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

cudaError_t read_wait_timeouts(unsigned long long* out, bool reset) {
    cudaError_t e = cudaMemcpyFromSymbol(out, g_wait_timeouts, sizeof(*out));
    if (e != cudaSuccess || !reset) return e;
    const unsigned long long zero = 0ull;
    return cudaMemcpyToSymbol(g_wait_timeouts, &zero, sizeof(zero));
}

}  // namespace coat
