// host_stream.cu -- the fused FP8 AdamW + DRE step over an optimizer state
// that lives in host memory (state offloading: the memory the FP8 state saves
// is what lets it sit in host memory at all).  The state and the gradient are
// streamed through a caller-provided device workspace in chunks; host->device
// copies, the step kernel and device->host copies of consecutive chunks run
// on three streams so that both copy directions overlap the compute.
#include <cstdint>
#include <cuda_runtime.h>

#include "coat.h"
#include "coat_kernels.h"

namespace {

constexpr int kSlots = 3;             // chunks in flight
constexpr int64_t kChunkQuantum = 4096;  // chunk sizes are multiples of this (and of G)

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Device bytes of one chunk slot of `c` parameters: w 4c, g 2c, codes 2c, records 16c/G.
size_t slot_bytes(int64_t c, int32_t G) {
    return align256(4 * (size_t)c) + align256(2 * (size_t)c) + 2 * align256((size_t)c) +
           align256(16 * (size_t)((c + G - 1) / G));
}

bool is_host(const void* p) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return at.type == cudaMemoryTypeHost || at.type == cudaMemoryTypeUnregistered;
}

bool is_device_mem(const void* p) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return at.type == cudaMemoryTypeDevice;
}

}  // namespace

extern "C" {

size_t coat_fp8_adamw_step_host_workspace_bytes(int64_t chunk_params, int32_t G) {
    if (chunk_params < 1 || G < 1 || G > 256 || (G & (G - 1)) != 0) return 0;
    const int64_t c = (chunk_params + kChunkQuantum - 1) / kChunkQuantum * kChunkQuantum;
    return (size_t)kSlots * slot_bytes(c, G);
}

coat_status coat_fp8_adamw_step_host(float* w, const uint16_t* g, uint8_t* m_q, uint8_t* v_q,
                                     coat_group_meta* meta, int64_t n, int32_t G, float beta1,
                                     float beta2, float lr, float eps, float weight_decay,
                                     int64_t step, void* workspace, size_t workspace_bytes,
                                     void* stream) {
    coat_status st = coat::check_step_args(w, g, m_q, v_q, meta, n, G, beta1, beta2, lr, eps,
                                           weight_decay, step);
    if (st != COAT_OK) return st;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
        return workspace ? COAT_ERR_MISALIGNED : COAT_ERR_INVALID_ARG;
    if (!is_host(w) || !is_host(g) || !is_host(m_q) || !is_host(v_q) || !is_host(meta))
        return COAT_ERR_INVALID_ARG;
    if (!is_device_mem(workspace)) return COAT_ERR_NOT_DEVICE;
    // largest chunk (multiple of 4096) whose three slots fit the workspace
    int64_t c = (int64_t)(workspace_bytes / kSlots / (8 + 16.0 / G)) / kChunkQuantum * kChunkQuantum;
    const int64_t n_round = (n + kChunkQuantum - 1) / kChunkQuantum * kChunkQuantum;
    if (c > n_round) c = n_round;
    while (c >= kChunkQuantum && (size_t)kSlots * slot_bytes(c, G) > workspace_bytes) c -= kChunkQuantum;
    if (c < kChunkQuantum) return COAT_ERR_INVALID_ARG;  // workspace too small for one chunk

    coat::StepArgs proto;
    st = coat::make_step_args(beta1, beta2, lr, eps, weight_decay, step, proto);
    if (st != COAT_OK) return st;

    cudaStream_t caller = static_cast<cudaStream_t>(stream);
    cudaStream_t s[kSlots] = {nullptr, nullptr, nullptr};
    cudaEvent_t ready = nullptr;
    cudaError_t err = cudaEventCreateWithFlags(&ready, cudaEventDisableTiming);
    for (int i = 0; i < kSlots && err == cudaSuccess; ++i)
        err = cudaStreamCreateWithFlags(&s[i], cudaStreamNonBlocking);
    // the chunks start after everything already queued on the caller's stream
    if (err == cudaSuccess) err = cudaEventRecord(ready, caller);
    for (int i = 0; i < kSlots && err == cudaSuccess; ++i) err = cudaStreamWaitEvent(s[i], ready, 0);

    const size_t sb = slot_bytes(c, G);
    char* ws = static_cast<char*>(workspace);
    for (int64_t a0 = 0, ci = 0; a0 < n && err == cudaSuccess; a0 += c, ++ci) {
        const int64_t m = (n - a0 < c) ? n - a0 : c;
        const int64_t ga = a0 / G, gb = (a0 + m + G - 1) / G;
        const int slot = (int)(ci % kSlots);
        cudaStream_t cs = s[slot];
        char* base = ws + slot * sb;
        float* dw = reinterpret_cast<float*>(base);
        uint16_t* dg = reinterpret_cast<uint16_t*>(base + align256(4 * (size_t)c));
        uint8_t* dm = reinterpret_cast<uint8_t*>(base + align256(4 * (size_t)c) + align256(2 * (size_t)c));
        uint8_t* dv = dm + align256((size_t)c);
        float4* dmeta = reinterpret_cast<float4*>(dv + align256((size_t)c));
        const size_t mb = (size_t)m, gbytes = 16 * (size_t)(gb - ga);
        err = cudaMemcpyAsync(dw, w + a0, 4 * mb, cudaMemcpyHostToDevice, cs);
        if (err == cudaSuccess) err = cudaMemcpyAsync(dg, g + a0, 2 * mb, cudaMemcpyHostToDevice, cs);
        if (err == cudaSuccess) err = cudaMemcpyAsync(dm, m_q + a0, mb, cudaMemcpyHostToDevice, cs);
        if (err == cudaSuccess) err = cudaMemcpyAsync(dv, v_q + a0, mb, cudaMemcpyHostToDevice, cs);
        if (err == cudaSuccess) err = cudaMemcpyAsync(dmeta, meta + ga, gbytes, cudaMemcpyHostToDevice, cs);
        if (err == cudaSuccess) {
            coat::StepArgs a = proto;
            a.w = dw;
            a.g = dg;
            a.mq = dm;
            a.vq = dv;
            a.meta = dmeta;
            a.n = m;
            err = coat::launch_adamw_dre_step(a, G, cs);
        }
        if (err == cudaSuccess) err = cudaMemcpyAsync(w + a0, dw, 4 * mb, cudaMemcpyDeviceToHost, cs);
        if (err == cudaSuccess) err = cudaMemcpyAsync(m_q + a0, dm, mb, cudaMemcpyDeviceToHost, cs);
        if (err == cudaSuccess) err = cudaMemcpyAsync(v_q + a0, dv, mb, cudaMemcpyDeviceToHost, cs);
        if (err == cudaSuccess) err = cudaMemcpyAsync(meta + ga, dmeta, gbytes, cudaMemcpyDeviceToHost, cs);
    }
    // the call returns once the host buffers hold the result
    for (int i = 0; i < kSlots; ++i) {
        if (s[i]) {
            const cudaError_t e2 = cudaStreamSynchronize(s[i]);
            if (err == cudaSuccess) err = e2;
            cudaStreamDestroy(s[i]);
        }
    }
    if (ready) cudaEventDestroy(ready);
    return err == cudaSuccess ? COAT_OK : COAT_ERR_CUDA;
}

}  // extern "C"
