// host_static.cu -- the host-memory step (state offloading) for callers that
// cannot allocate device memory.
//
// coat_fp8_adamw_step_host streams the state through a workspace the caller
// allocates.  Some callers cannot make that allocation: a process whose
// caching allocator already holds the device memory it may use, code that
// must not call cudaMalloc / cudaFree (they can synchronize the whole device)
// in the middle of a step, or a runtime that fixes its device footprint at
// start-up.  This entry point streams through a fixed scratch buffer that is a
// file-scope __device__ array of this translation unit instead: the CUDA
// runtime reserves it on a device when it loads this file's module there, and
// the call itself allocates nothing.
#include <cstdint>
#include <cuda_runtime.h>

#include "coat.h"
#include "coat_kernels.h"

namespace {

constexpr int64_t kChunkQuantum = 4096;  // chunk sizes are multiples of this (and of G)

// The scratch of one chunk; nothing in it has to start at zero (every byte the
// kernel reads is copied in by the same call first).
__device__ __align__(256) unsigned char g_static_scratch[COAT_STATIC_SCRATCH_BYTES];

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Device bytes of one chunk of `c` parameters: w 4c, g 2c, codes 2c, records 16c/G.
size_t chunk_bytes(int64_t c, int32_t G) {
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

// The scratch's address on the current device (the array's name is only a
// host-side stand-in).  It is looked up on every call: a lookup allocates
// nothing, and a cached address would outlive a device reset, after which the
// module is loaded again and the array may sit elsewhere.  The first lookup
// on a device may load this module there.
cudaError_t scratch_on_current_device(unsigned char** out) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return e;
    *out = static_cast<unsigned char*>(p);
    return cudaSuccess;
}

// A stream that belongs to another device than the current one would queue
// the copies before the launch fails: refuse it first.
bool stream_on_current_device(cudaStream_t s) {
    if (s == nullptr) return true;   // the legacy default stream of the current device
    int cur = -1, dev = -1;
    if (cudaGetDevice(&cur) != cudaSuccess || cudaStreamGetDevice(s, &dev) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return cur == dev;
}

}  // namespace

extern "C" {

coat_status coat_fp8_adamw_step_host_static(float* w, const uint16_t* g, uint8_t* m_q,
                                            uint8_t* v_q, coat_group_meta* meta, int64_t n,
                                            int32_t G, float beta1, float beta2, float lr,
                                            float eps, float weight_decay, int64_t step,
                                            int64_t chunk_params, void* stream) {
    coat_status st = coat::check_step_args(w, g, m_q, v_q, meta, n, G, beta1, beta2, lr, eps,
                                           weight_decay, step);
    if (st != COAT_OK) return st;
    if (chunk_params < 0) return COAT_ERR_INVALID_ARG;
    // every parameter needs more than one byte of scratch: this also bounds the rounding below
    if (chunk_params > (int64_t)COAT_STATIC_SCRATCH_BYTES) return COAT_ERR_SCRATCH_LIMIT;
    int64_t c;
    if (chunk_params == 0) {  // the largest chunk that fits
        c = (int64_t)COAT_STATIC_SCRATCH_BYTES / 8 / kChunkQuantum * kChunkQuantum;
        while (c >= kChunkQuantum && chunk_bytes(c, G) > COAT_STATIC_SCRATCH_BYTES) c -= kChunkQuantum;
    } else {
        c = (chunk_params + kChunkQuantum - 1) / kChunkQuantum * kChunkQuantum;
        if (chunk_bytes(c, G) > COAT_STATIC_SCRATCH_BYTES) return COAT_ERR_SCRATCH_LIMIT;
    }
    const int64_t n_round = (n + kChunkQuantum - 1) / kChunkQuantum * kChunkQuantum;
    if (c > n_round) c = n_round;
    if (!is_host(w) || !is_host(g) || !is_host(m_q) || !is_host(v_q) || !is_host(meta))
        return COAT_ERR_INVALID_ARG;
    coat::StepArgs proto;
    st = coat::make_step_args(beta1, beta2, lr, eps, weight_decay, step, proto);
    if (st != COAT_OK) return st;
    if (!stream_on_current_device(static_cast<cudaStream_t>(stream))) return COAT_ERR_INVALID_ARG;
    unsigned char* scratch = nullptr;
    cudaError_t err = scratch_on_current_device(&scratch);
    if (err != cudaSuccess) return COAT_ERR_CUDA;

    // One chunk at a time on the caller's stream: copies in, the step, copies
    // out.  Stream order keeps a chunk's copies in from overwriting the
    // scratch before the previous chunk's copies out have read it.
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    float* dw = reinterpret_cast<float*>(scratch);
    uint16_t* dg = reinterpret_cast<uint16_t*>(scratch + align256(4 * (size_t)c));
    uint8_t* dm = scratch + align256(4 * (size_t)c) + align256(2 * (size_t)c);
    uint8_t* dv = dm + align256((size_t)c);
    float4* dmeta = reinterpret_cast<float4*>(dv + align256((size_t)c));
    for (int64_t a0 = 0; a0 < n && err == cudaSuccess; a0 += c) {
        const int64_t m = (n - a0 < c) ? n - a0 : c;
        const int64_t ga = a0 / G, gb = (a0 + m + G - 1) / G;
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
    const cudaError_t e2 = cudaStreamSynchronize(cs);
    if (err == cudaSuccess) err = e2;
    return err == cudaSuccess ? COAT_OK : COAT_ERR_CUDA;
}

}  // extern "C"
