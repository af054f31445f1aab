// coat_kernels.h -- internal launch interface between the C ABI (coat_abi.cu)
// and the kernels.  Not part of the public header.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace coat {

struct StepArgs {
    float* w;
    const uint16_t* g;
    uint8_t* mq;
    uint8_t* vq;
    float4* meta;
    int64_t n;
    float beta1, beta2;
    float omb1, omb2;  // 1 - beta (exact in fp32 for beta in [0.5, 1))
    float c1;          // lr / (1 - beta1^t)
    float c2;          // 1 / (1 - beta2^t)
    float eps;
    float decay;       // 1 - lr * weight_decay
    // the update's denominator scaled by -1/c1: -(sqrt(v c2) + eps) / c1 =
    // sqrt(v) sq + ep, so that w - c1 m / (sqrt(v c2) + eps) = w + m / (sqrt(v) sq + ep)
    // (lr = 0: sq = 1, ep = +inf, and the update term is 0)
    float sq;          // -sqrt(c2) / c1
    float ep;          // -eps / c1
};

struct QuantArgs {
    const float* x;
    uint8_t* q;
    float* scale;
    float* k;
    int64_t n;
};

struct DequantArgs {
    const uint8_t* q;
    const float* scale;
    const float* k;
    float* x;
    int64_t n;
};

cudaError_t launch_adamw_dre_step(const StepArgs& a, int G, cudaStream_t stream);
// the step kernel's float64-recomputation counters on the current device
cudaError_t read_recompute_counts(unsigned long long out[2], bool reset);

}  // namespace coat

#include "coat.h"

namespace coat {

// argument checks shared by the device-buffer and host-buffer steps (coat_abi.cu)
coat_status check_step_args(const float* w, const uint16_t* g, const uint8_t* m_q,
                            const uint8_t* v_q, const coat_group_meta* meta, int64_t n, int32_t G,
                            float beta1, float beta2, float lr, float eps, float weight_decay,
                            int64_t step);
// per-launch constants of the step (everything but the buffers)
coat_status make_step_args(float beta1, float beta2, float lr, float eps, float weight_decay,
                           int64_t step, StepArgs& a);
struct ActArgs {
    const uint16_t* x;   // M x N bf16, row-major
    int64_t M, N;
    uint8_t* q;          // M x N codes
    uint8_t* qt;         // N x M codes (may be null)
    float* scale;        // M x N/G
};

struct LinArgs {
    const uint8_t* xq;   // M x K E4M3 codes, row-major
    const uint8_t* wq;   // N x K E4M3 codes, row-major
    float sx, sw;        // per-tensor scales of X and W
    int64_t M, N, K;
    uint8_t* q;          // M x N output codes
    float* scale;        // M x N/G output group scales
    float* y;            // M x N float32 output before quantization (may be null)
};

cudaError_t launch_dre_quantize(const QuantArgs& a, int G, cudaStream_t stream);
cudaError_t launch_linear_fp8(const LinArgs& a, int G, cudaStream_t stream);
// bounded waits in the library's kernels that gave up, on the current device
cudaError_t read_wait_timeouts(unsigned long long* out, bool reset);
cudaError_t launch_act_quant(const ActArgs& a, int G, cudaStream_t stream);
cudaError_t launch_absmax_quantize(const QuantArgs& a, int G, cudaStream_t stream);
cudaError_t launch_dre_dequantize(const DequantArgs& a, int G, cudaStream_t stream);

}  // namespace coat
