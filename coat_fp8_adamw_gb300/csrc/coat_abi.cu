// coat_abi.cu -- the extern "C" entry points declared in include/coat.h:
// argument validation, per-launch constants (bias corrections), and the
// dispatch to the templated kernels.  No allocation, no state, no host sync.
#include <cmath>
#include <cstdint>
#include <cuda_runtime.h>

#include "coat.h"
#include "coat_kernels.h"

namespace {

bool pow2_group(int32_t G) { return G >= 1 && G <= 256 && (G & (G - 1)) == 0; }
bool size_ok(int64_t n) { return n >= 1 && n <= COAT_MAX_N; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + nb && b0 < a0 + na;
}

// Device memory of the current device, or managed memory.  Host memory is
// refused even where the GPU could reach it, since the kernels assume HBM,
// and so is another device's memory: the kernels launch on the current one.
bool is_device(const void* p) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();  // clear the sticky-free error state of this query
        return false;
    }
    if (at.type == cudaMemoryTypeManaged) return true;
    if (at.type != cudaMemoryTypeDevice) return false;
    int cur = -1;
    if (cudaGetDevice(&cur) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return at.device == cur;
}

coat_status from_cuda(cudaError_t e) { return e == cudaSuccess ? COAT_OK : COAT_ERR_CUDA; }

int64_t num_groups(int64_t n, int32_t G) { return (n + G - 1) / G; }


}  // namespace

namespace coat {

// Checks shared by the device- and host-buffer steps (everything but where the
// buffers live), and the per-launch constants.
coat_status check_step_args(const float* w, const uint16_t* g, const uint8_t* m_q,
                            const uint8_t* v_q, const coat_group_meta* meta, int64_t n, int32_t G,
                            float beta1, float beta2, float lr, float eps, float weight_decay,
                            int64_t step) {
    if (!w || !g || !m_q || !v_q || !meta || !size_ok(n) || step < 1) return COAT_ERR_INVALID_ARG;
    if (!pow2_group(G)) return COAT_ERR_UNSUPPORTED_G;
    if (!aligned16(w) || !aligned16(g) || !aligned16(m_q) || !aligned16(v_q) || !aligned16(meta))
        return COAT_ERR_MISALIGNED;
    if (!std::isfinite(beta1) || !std::isfinite(beta2) || !std::isfinite(lr) ||
        !std::isfinite(eps) || !std::isfinite(weight_decay) || beta1 < 0.0f || beta1 >= 1.0f ||
        beta2 < 0.0f || beta2 >= 1.0f || lr < 0.0f || !(eps > 0.0f) || weight_decay < 0.0f)
        return COAT_ERR_INVALID_ARG;
    const size_t nb = (size_t)n;
    const size_t ng = (size_t)num_groups(n, G);
    if (overlaps(g, 2 * nb, w, 4 * nb) || overlaps(g, 2 * nb, m_q, nb) ||
        overlaps(g, 2 * nb, v_q, nb) || overlaps(g, 2 * nb, meta, 16 * ng) ||
        overlaps(w, 4 * nb, m_q, nb) || overlaps(w, 4 * nb, v_q, nb) ||
        overlaps(w, 4 * nb, meta, 16 * ng) || overlaps(m_q, nb, v_q, nb) ||
        overlaps(m_q, nb, meta, 16 * ng) || overlaps(v_q, nb, meta, 16 * ng))
        return COAT_ERR_INVALID_ARG;
    return COAT_OK;
}

// Bias corrections 1 - beta^t once per launch in double; the kernel gets
// lr / (1 - beta1^t), 1 / (1 - beta2^t), 1 - beta and 1 - lr wd as floats.
coat_status make_step_args(float beta1, float beta2, float lr, float eps, float weight_decay,
                           int64_t step, StepArgs& a) {
    const double b1 = beta1, b2 = beta2;
    const double bc1 = 1.0 - std::pow(b1, (double)step);
    const double bc2 = 1.0 - std::pow(b2, (double)step);
    if (!(bc1 > 0.0) || !(bc2 > 0.0)) return COAT_ERR_INVALID_ARG;
    a.beta1 = beta1;
    a.beta2 = beta2;
    a.omb1 = (float)(1.0 - b1);
    a.omb2 = (float)(1.0 - b2);
    a.c1 = (float)((double)lr / bc1);
    a.c2 = (float)(1.0 / bc2);
    a.eps = eps;
    a.decay = (float)(1.0 - (double)lr * (double)weight_decay);
    const double c1 = (double)lr / bc1;
    if (c1 > 0.0) {
        a.sq = (float)(-std::sqrt(1.0 / bc2) / c1);
        a.ep = (float)(-(double)eps / c1);
    } else {
        a.sq = 1.0f;
        a.ep = INFINITY;
    }
    return COAT_OK;
}

}  // namespace coat

extern "C" {

coat_status coat_fp8_adamw_step(float* w, const uint16_t* g, uint8_t* m_q, uint8_t* v_q,
                                coat_group_meta* meta, int64_t n, int32_t G, float beta1,
                                float beta2, float lr, float eps, float weight_decay,
                                int64_t step, void* stream) {
    coat_status st = coat::check_step_args(w, g, m_q, v_q, meta, n, G, beta1, beta2, lr, eps,
                                           weight_decay, step);
    if (st != COAT_OK) return st;
    if (!is_device(w) || !is_device(g) || !is_device(m_q) || !is_device(v_q) || !is_device(meta))
        return COAT_ERR_NOT_DEVICE;
    coat::StepArgs a;
    st = coat::make_step_args(beta1, beta2, lr, eps, weight_decay, step, a);
    if (st != COAT_OK) return st;
    a.w = w;
    a.g = g;
    a.mq = m_q;
    a.vq = v_q;
    a.meta = reinterpret_cast<float4*>(meta);
    a.n = n;
    return from_cuda(coat::launch_adamw_dre_step(a, G, static_cast<cudaStream_t>(stream)));
}

coat_status coat_dre_quantize(const float* x, int64_t n, int32_t G, uint8_t* q, float* scale,
                              float* k, void* stream) {
    if (!x || !q || !scale || !k || !size_ok(n)) return COAT_ERR_INVALID_ARG;
    if (!pow2_group(G)) return COAT_ERR_UNSUPPORTED_G;
    if (!aligned16(x) || !aligned16(q) || !aligned16(scale) || !aligned16(k))
        return COAT_ERR_MISALIGNED;
    const size_t nb = (size_t)n, ng = (size_t)num_groups(n, G);
    if (overlaps(x, 4 * nb, q, nb) || overlaps(x, 4 * nb, scale, 4 * ng) ||
        overlaps(x, 4 * nb, k, 4 * ng) || overlaps(q, nb, scale, 4 * ng) ||
        overlaps(q, nb, k, 4 * ng) || overlaps(scale, 4 * ng, k, 4 * ng))
        return COAT_ERR_INVALID_ARG;
    if (!is_device(x) || !is_device(q) || !is_device(scale) || !is_device(k))
        return COAT_ERR_NOT_DEVICE;
    coat::QuantArgs a{x, q, scale, k, n};
    return from_cuda(coat::launch_dre_quantize(a, G, static_cast<cudaStream_t>(stream)));
}

coat_status coat_fp8_quantize_absmax(const float* x, int64_t n, int32_t G, uint8_t* q, float* scale,
                                     void* stream) {
    if (!x || !q || !scale || !size_ok(n)) return COAT_ERR_INVALID_ARG;
    if (!pow2_group(G)) return COAT_ERR_UNSUPPORTED_G;
    if (!aligned16(x) || !aligned16(q) || !aligned16(scale)) return COAT_ERR_MISALIGNED;
    const size_t nb = (size_t)n, ng = (size_t)num_groups(n, G);
    if (overlaps(x, 4 * nb, q, nb) || overlaps(x, 4 * nb, scale, 4 * ng) ||
        overlaps(q, nb, scale, 4 * ng))
        return COAT_ERR_INVALID_ARG;
    if (!is_device(x) || !is_device(q) || !is_device(scale)) return COAT_ERR_NOT_DEVICE;
    coat::QuantArgs a{x, q, scale, nullptr, n};
    return from_cuda(coat::launch_absmax_quantize(a, G, static_cast<cudaStream_t>(stream)));
}

coat_status coat_act_quantize_fp8(const uint16_t* x, int64_t M, int64_t N, int32_t G, uint8_t* q,
                                  uint8_t* qt, float* scale, void* stream) {
    if (!x || !q || !scale || M < 1 || N < 1) return COAT_ERR_INVALID_ARG;
    if (G < 4 || G > 128 || (G & (G - 1)) != 0) return COAT_ERR_UNSUPPORTED_G;
    if (M % 16 != 0 || N % 16 != 0 || N % G != 0) return COAT_ERR_INVALID_ARG;
    if (M > 65535LL * 64 || N / 128 >= (1LL << 31)) return COAT_ERR_INVALID_ARG;   // grid limits
    if (!aligned16(x) || !aligned16(q) || !aligned16(scale) || (qt && !aligned16(qt)))
        return COAT_ERR_MISALIGNED;
    const size_t ne = (size_t)M * (size_t)N, ns = ne / (size_t)G;
    if (overlaps(x, 2 * ne, q, ne) || overlaps(x, 2 * ne, scale, 4 * ns) ||
        overlaps(q, ne, scale, 4 * ns) ||
        (qt && (overlaps(qt, ne, x, 2 * ne) || overlaps(qt, ne, q, ne) || overlaps(qt, ne, scale, 4 * ns))))
        return COAT_ERR_INVALID_ARG;
    if (!is_device(x) || !is_device(q) || !is_device(scale) || (qt && !is_device(qt)))
        return COAT_ERR_NOT_DEVICE;
    coat::ActArgs a{x, M, N, q, qt, scale};
    return from_cuda(coat::launch_act_quant(a, G, static_cast<cudaStream_t>(stream)));
}

coat_status coat_fp8_linear_group_quantize(const uint8_t* xq, float sx, const uint8_t* wq,
                                           float sw, int64_t M, int64_t N, int64_t K, int32_t G,
                                           uint8_t* q, float* scale, float* y, void* stream) {
    if (!xq || !wq || !q || !scale || M < 1 || N < 1 || K < 1) return COAT_ERR_INVALID_ARG;
    if (!(sx > 0.0f) || !(sw > 0.0f) || !std::isfinite(sx) || !std::isfinite(sw))
        return COAT_ERR_INVALID_ARG;
    if (G < 8 || G > 128 || (G & (G - 1)) != 0) return COAT_ERR_UNSUPPORTED_G;
    if (N % 16 != 0 || N % G != 0 || K % 16 != 0) return COAT_ERR_INVALID_ARG;
    if (M >= (1LL << 31) || N >= (1LL << 31) || K >= (1LL << 31)) return COAT_ERR_INVALID_ARG;
    if (!aligned16(xq) || !aligned16(wq) || !aligned16(q) || !aligned16(scale) || (y && !aligned16(y)))
        return COAT_ERR_MISALIGNED;
    const size_t nx = (size_t)M * (size_t)K, nw = (size_t)N * (size_t)K;
    const size_t ny = (size_t)M * (size_t)N, ns = 4 * (ny / (size_t)G);
    const void* out[3] = {q, scale, y};
    const size_t nout[3] = {ny, ns, 4 * ny};
    for (int i = 0; i < 3; ++i) {
        if (!out[i]) continue;
        if (overlaps(out[i], nout[i], xq, nx) || overlaps(out[i], nout[i], wq, nw)) return COAT_ERR_INVALID_ARG;
        for (int j = i + 1; j < 3; ++j)
            if (out[j] && overlaps(out[i], nout[i], out[j], nout[j])) return COAT_ERR_INVALID_ARG;
    }
    if (!is_device(xq) || !is_device(wq) || !is_device(q) || !is_device(scale) || (y && !is_device(y)))
        return COAT_ERR_NOT_DEVICE;
    coat::LinArgs a{xq, wq, sx, sw, M, N, K, q, scale, y};
    return from_cuda(coat::launch_linear_fp8(a, G, static_cast<cudaStream_t>(stream)));
}

coat_status coat_dre_dequantize(const uint8_t* q, const float* scale, const float* k, int64_t n,
                                int32_t G, float* x, void* stream) {
    if (!x || !q || !scale || !k || !size_ok(n)) return COAT_ERR_INVALID_ARG;
    if (!pow2_group(G)) return COAT_ERR_UNSUPPORTED_G;
    if (!aligned16(x) || !aligned16(q) || !aligned16(scale) || !aligned16(k))
        return COAT_ERR_MISALIGNED;
    const size_t nb = (size_t)n, ng = (size_t)num_groups(n, G);
    if (overlaps(x, 4 * nb, q, nb) || overlaps(x, 4 * nb, scale, 4 * ng) ||
        overlaps(x, 4 * nb, k, 4 * ng))
        return COAT_ERR_INVALID_ARG;
    if (!is_device(x) || !is_device(q) || !is_device(scale) || !is_device(k))
        return COAT_ERR_NOT_DEVICE;
    coat::DequantArgs a{q, scale, k, x, n};
    return from_cuda(coat::launch_dre_dequantize(a, G, static_cast<cudaStream_t>(stream)));
}

coat_status coat_kernel_wait_timeouts(uint64_t* count, int32_t reset) {
    if (!count) return COAT_ERR_INVALID_ARG;
    unsigned long long c = 0ull;
    if (coat::read_wait_timeouts(&c, reset != 0) != cudaSuccess) return COAT_ERR_CUDA;
    *count = c;
    return COAT_OK;
}

coat_status coat_exact_recompute_counts(uint64_t counts[2], int32_t reset) {
    if (!counts) return COAT_ERR_INVALID_ARG;
    unsigned long long c[2] = {0ull, 0ull};
    const cudaError_t e = coat::read_recompute_counts(c, reset != 0);
    if (e != cudaSuccess) return COAT_ERR_CUDA;
    counts[0] = c[0];
    counts[1] = c[1];
    return COAT_OK;
}

const char* coat_status_string(coat_status s) {
    switch (s) {
        case COAT_OK: return "ok";
        case COAT_ERR_INVALID_ARG: return "invalid argument";
        case COAT_ERR_MISALIGNED: return "pointer not 16-byte aligned";
        case COAT_ERR_UNSUPPORTED_G: return "group size must be a power of two in [1, 256]";
        case COAT_ERR_CUDA: return "CUDA launch or runtime error";
        case COAT_ERR_NOT_DEVICE: return "pointer is not device memory";
        case COAT_ERR_SCRATCH_LIMIT: return "request exceeds the library's static scratch";
    }
    return "unknown status";
}

double coat_r_e4m3(void) { return 448.0 * 512.0; }

int32_t coat_version(void) { return 200; }

}  // extern "C"
