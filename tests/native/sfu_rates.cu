// Throughput of the SFU instructions the fast path uses, on the device this
// runs on: 8 independent chains of one instruction per thread, 4 CTAs of 512
// threads per SM, 4096 rounds; prints results per SM and clock (at the
// device's nominal clock) for each instruction, one "name rate" line each.
// Every thread writes one float, so the output buffer holds exactly
// grid x block floats.
#include <cstdio>
#include <cuda_runtime.h>

namespace {
constexpr int kRounds = 4096;
constexpr int kChains = 8;

template <int OP>
__device__ __forceinline__ float op(float x) {
    float y;
    if constexpr (OP == 0) asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    else if constexpr (OP == 1) asm volatile("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    else if constexpr (OP == 2) asm volatile("sqrt.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    else asm volatile("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <int OP>
__global__ void chains(float* out, float seed) {
    float c[kChains];
#pragma unroll
    for (int i = 0; i < kChains; ++i) c[i] = seed + 0.01f * (threadIdx.x & 7) + 0.001f * i;
    for (int r = 0; r < kRounds; ++r) {
#pragma unroll
        for (int i = 0; i < kChains; ++i) c[i] = op<OP>(c[i]);
    }
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < kChains; ++i) s += c[i];
    out[blockIdx.x * blockDim.x + threadIdx.x] = s;
}

template <int OP>
int run(const char* name, float* out, int sms, int clk_khz) {
    const int blocks = sms * 4, threads = 512;
    chains<OP><<<blocks, threads>>>(out, 0.37f);
    cudaEvent_t a, b;
    cudaEventCreate(&a);
    cudaEventCreate(&b);
    cudaEventRecord(a);
    chains<OP><<<blocks, threads>>>(out, 0.37f);
    cudaEventRecord(b);
    if (cudaEventSynchronize(b) != cudaSuccess) return 1;
    float ms = 0.0f;
    cudaEventElapsedTime(&ms, a, b);
    const double ops = (double)blocks * threads * kRounds * kChains;
    std::printf("%s %.2f\n", name, ops / (ms * 1e-3) / sms / (clk_khz * 1e3));
    cudaEventDestroy(a);
    cudaEventDestroy(b);
    return cudaGetLastError() == cudaSuccess ? 0 : 1;
}
}  // namespace

int main() {
    int sms = 0, clk = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
    cudaDeviceGetAttribute(&clk, cudaDevAttrClockRate, 0);
    float* out = nullptr;
    if (cudaMalloc(&out, sizeof(float) * sms * 4 * 512) != cudaSuccess) return 1;
    int bad = run<0>("ex2", out, sms, clk) | run<1>("lg2", out, sms, clk) |
              run<2>("sqrt", out, sms, clk) | run<3>("rsqrt", out, sms, clk);
    cudaFree(out);
    return bad;
}
