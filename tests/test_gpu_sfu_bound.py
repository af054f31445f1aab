"""The relative error of the SFU exp2 (PTX ex2.approx.ftz.f32) that the step
kernel's fast-path error bound assumes (its constant kEx2Err, read from the
kernel source): no larger than that for every fp32 input whose result is a
normal float, over the arguments the fast path gives it
(the fractional part of a scale exponent, and L(q)/k <= 0 for a stored code).

The check is exhaustive: a small probe, compiled here with nvcc, evaluates
the instruction for every fp32 value in (-126, 9] and compares it with the
double-precision exp2 of the same input.  The open end stops one float above
-126, whose exact result 2^-126 is the smallest normal float.
"""
import ctypes
import math
import os
import shutil
import struct
import subprocess

import pytest

from _kernel_consts import kernel_ex2_bound

PROBE = r"""
#include <cstdint>
#include <cuda_runtime.h>

__device__ __forceinline__ float ex2_ftz(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// every float with bit pattern in [b0, b1] (one sign): max relative error as
// the bits of a non-negative double (ordered like the value)
__global__ void probe(uint32_t b0, uint32_t b1, unsigned long long* worst) {
    unsigned long long local = 0ull;
    const uint64_t total = (uint64_t)b1 - b0 + 1;
    for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < total;
         i += (uint64_t)gridDim.x * blockDim.x) {
        const float x = __uint_as_float(b0 + (uint32_t)i);
        const double ref = exp2((double)x);
        const double rel = fabs((double)ex2_ftz(x) - ref) / ref;
        const unsigned long long bits = (unsigned long long)__double_as_longlong(rel);
        local = bits > local ? bits : local;
    }
    atomicMax(worst, local);
}

extern "C" double max_rel_err(uint32_t b0, uint32_t b1) {
    unsigned long long* d = nullptr;
    if (cudaMalloc(&d, sizeof(*d)) != cudaSuccess) return -1.0;
    cudaMemset(d, 0, sizeof(*d));
    probe<<<152 * 16, 256>>>(b0, b1, d);
    unsigned long long h = 0ull;
    const cudaError_t e = cudaMemcpy(&h, d, sizeof(h), cudaMemcpyDeviceToHost);
    cudaFree(d);
    if (e != cudaSuccess) return -1.0;
    double r;
    static_assert(sizeof(r) == sizeof(h), "");
    __builtin_memcpy(&r, &h, sizeof(r));
    return r;
}
"""


def _f32_bits(v):
    return struct.unpack("<I", struct.pack("<f", v))[0]


def test_kernel_bound_is_a_power_of_two():
    b = kernel_ex2_bound()
    assert math.frexp(b)[0] == 0.5 and 2.0 ** -24 < b <= 2.0 ** -21


@pytest.mark.gpu
def test_ex2_approx_ftz_relative_error_within_kernel_bound(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    src = tmp_path / "probe.cu"
    lib = tmp_path / "probe.so"
    src.write_text(PROBE)
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-shared",
                    "-Xcompiler", "-fPIC", "-o", str(lib), str(src)], check=True,
                   capture_output=True)
    L = ctypes.CDLL(str(lib))
    L.max_rel_err.argtypes = [ctypes.c_uint32, ctypes.c_uint32]
    L.max_rel_err.restype = ctypes.c_double
    # [0, 9] and (-126, -0]: exact results from just above 2^-126 to 2^9
    worst_pos = L.max_rel_err(0, _f32_bits(9.0))
    worst_neg = L.max_rel_err(0x80000000, _f32_bits(-126.0) - 1)
    assert worst_pos >= 0.0 and worst_neg >= 0.0, "the probe failed to run"
    worst = max(worst_pos, worst_neg)
    bound = kernel_ex2_bound()
    print("max relative error of ex2.approx.ftz.f32: 2^%.3f (bound 2^%g)"
          % (math.log2(worst), math.log2(bound)))
    assert worst <= bound
