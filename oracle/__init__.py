"""Plain float64 CPU oracle for the fused FP8 AdamW + DRE step.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import this package.  The
product path (the CUDA library and its binding) never loads it and shares no
code with it.

The arithmetic lives in ``coat_oracle.c`` (plain C, float64, libm ``pow`` /
``log``; no fast-math, no FMA contraction) and follows the COAT paper-review
page (xllm-io, "COAT: Compressing Optimizer States and Activation for
Memory-Efficient FP8 Training"), section 3 core formulas: the FP8
quantization equation, the AdamW update rule and the Dynamic Range Expansion
equations.  This module only marshals numpy arrays through ctypes.

Every function here is pinned by ``tests/test_oracle_*.py`` against things
other than itself: the E4M3 table of the OCP FP8 format and torch's
float8_e4m3fn conversion, the scalar closed form of AdamW under constant
gradients and torch's AdamW, the identity R_X^k = R_E4M3, bisection for k,
and hand-computed worked examples under ``tests/golden/``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "coat_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libcoat_oracle.so")

#: the library's reading of the page's R_E4M3: max finite / min subnormal
R_E4M3_DEFAULT = 448.0 / 2.0 ** -9
#: the alternative reading: max finite / min normal
R_E4M3_MIN_NORMAL = 448.0 / 2.0 ** -6

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C11, -O2, no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-pthread",
           "-ffp-contract=off", "-fno-fast-math", "-D_GNU_SOURCE",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        # COAT_ORACLE_LIB lets the oracle's own mutation test load a deliberately
        # broken build of coat_oracle.c in a subprocess
        override = os.environ.get("COAT_ORACLE_LIB")
        lib = ctypes.CDLL(override if override else build())
        c_f32p = ctypes.POINTER(ctypes.c_float)
        c_f64p = ctypes.POINTER(ctypes.c_double)
        c_u8p = ctypes.POINTER(ctypes.c_uint8)
        c_u16p = ctypes.POINTER(ctypes.c_uint16)
        i64, i32, f32, f64 = ctypes.c_int64, ctypes.c_int32, ctypes.c_float, ctypes.c_double
        lib.coat_oracle_e4m3_decode.argtypes = [ctypes.c_int]
        lib.coat_oracle_e4m3_decode.restype = f64
        lib.coat_oracle_e4m3_encode.argtypes = [f64]
        lib.coat_oracle_e4m3_encode.restype = ctypes.c_int
        lib.coat_oracle_dre_group.argtypes = [c_f32p, i64, f64, c_f64p, c_f64p, c_f32p,
                                              c_f32p, c_f64p, c_u8p]
        lib.coat_oracle_dre_group.restype = ctypes.c_int
        lib.coat_oracle_dre_quantize.argtypes = [c_f32p, i64, i32, f64, c_u8p, c_f32p, c_f32p,
                                                 ctypes.c_int]
        lib.coat_oracle_dre_quantize.restype = ctypes.c_int
        lib.coat_oracle_absmax_quantize.argtypes = [c_f32p, i64, i32, c_u8p, c_f32p, ctypes.c_int]
        lib.coat_oracle_absmax_quantize.restype = ctypes.c_int
        lib.coat_oracle_dre_dequantize.argtypes = [c_u8p, c_f32p, c_f32p, i64, i32, c_f32p,
                                                   ctypes.c_int]
        lib.coat_oracle_dre_dequantize.restype = ctypes.c_int
        lib.coat_oracle_adamw_step.argtypes = [c_f32p, c_u16p, c_u8p, c_u8p, c_f32p, i64, i32,
                                               f32, f32, f32, f32, f32, i64, f64, ctypes.c_int]
        lib.coat_oracle_adamw_step.restype = ctypes.c_int
        lib.coat_oracle_threads.argtypes = [ctypes.c_int]
        lib.coat_oracle_threads.restype = ctypes.c_int
        _lib = lib
        return lib


def _ptr(a: np.ndarray, ctype):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def threads(nthreads: int = 0) -> int:
    """Number of host threads the oracle uses for ``nthreads`` (0 = all online cores)."""
    return int(_load().coat_oracle_threads(nthreads))


def e4m3_decode(code: int) -> float:
    """Value of one E4M3 code (bit definition: bias 7, subnormals, NaN at 0x7F/0xFF)."""
    return float(_load().coat_oracle_e4m3_decode(int(code)))


def e4m3_decode_all() -> np.ndarray:
    """Values of all 256 codes, indexed by code."""
    lib = _load()
    return np.array([lib.coat_oracle_e4m3_decode(c) for c in range(256)], dtype=np.float64)


def e4m3_encode(y: float) -> int:
    """Nearest finite E4M3 code (ties to even mantissa, saturating, zero -> 0x00)."""
    return int(_load().coat_oracle_e4m3_encode(float(y)))


def e4m3_encode_array(y: np.ndarray) -> np.ndarray:
    lib = _load()
    flat = np.asarray(y, dtype=np.float64).ravel()
    return np.array([lib.coat_oracle_e4m3_encode(float(v)) for v in flat],
                    dtype=np.uint8).reshape(np.shape(y))


def dre_group(x: np.ndarray, R: float = R_E4M3_DEFAULT) -> dict:
    """Everything the oracle computes for one group of fp32 values.

    Returns k before any cap (``k_formula``), after the cap and the S-range
    guard (``k_exact``), the stored fp32 ``k`` and ``S``, the expanded and
    scaled values ``y`` = f(x)/S in float64, and the codes ``q``.
    """
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float32)
    n = x.size
    kf = ctypes.c_double()
    ke = ctypes.c_double()
    k32 = ctypes.c_float()
    s32 = ctypes.c_float()
    y = np.zeros(n, dtype=np.float64)
    q = np.zeros(n, dtype=np.uint8)
    rc = lib.coat_oracle_dre_group(_ptr(x, ctypes.c_float), n, float(R), ctypes.byref(kf),
                                   ctypes.byref(ke), ctypes.byref(k32), ctypes.byref(s32),
                                   _ptr(y, ctypes.c_double), _ptr(q, ctypes.c_uint8))
    if rc != 0:
        raise ValueError("oracle dre_group: bad arguments")
    return {"k_formula": kf.value, "k_exact": ke.value, "k": np.float32(k32.value),
            "S": np.float32(s32.value), "y": y, "q": q}


def dre_quantize(x: np.ndarray, G: int, R: float = R_E4M3_DEFAULT, nthreads: int = 0):
    """Per-group DRE + E4M3 quantization of a flat fp32 buffer -> (q, S, k)."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float32).ravel()
    n = x.size
    ng = (n + G - 1) // G
    q = np.zeros(n, dtype=np.uint8)
    S = np.zeros(ng, dtype=np.float32)
    k = np.zeros(ng, dtype=np.float32)
    rc = lib.coat_oracle_dre_quantize(_ptr(x, ctypes.c_float), n, int(G), float(R),
                                      _ptr(q, ctypes.c_uint8), _ptr(S, ctypes.c_float),
                                      _ptr(k, ctypes.c_float), int(nthreads))
    if rc != 0:
        raise ValueError("oracle dre_quantize: bad arguments")
    return q, S, k


def absmax_quantize(x: np.ndarray, G: int, nthreads: int = 0):
    """Per-group FP8 quantization without the expansion -> (q, S): S = max|x| / 448
    rounded to float, q = E4M3(x / S) (section 3, FP8 quantization equation)."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float32).ravel()
    n = x.size
    ng = (n + G - 1) // G
    q = np.zeros(n, dtype=np.uint8)
    S = np.zeros(ng, dtype=np.float32)
    rc = lib.coat_oracle_absmax_quantize(_ptr(x, ctypes.c_float), n, int(G),
                                         _ptr(q, ctypes.c_uint8), _ptr(S, ctypes.c_float),
                                         int(nthreads))
    if rc != 0:
        raise ValueError("oracle absmax_quantize: bad arguments")
    return q, S


def act_quantize(x_bf16_bits: np.ndarray, G: int, nthreads: int = 0):
    """Per-group (1 x G) FP8 quantization of an M x N bf16 activation (raw bits)
    -> (q [M, N], qt [N, M], S [M, N/G]): each row split into groups of G
    columns, quantized like :func:`absmax_quantize`; qt is q transposed."""
    M, N = x_bf16_bits.shape
    if N % G:
        raise ValueError("oracle act_quantize: N must be a multiple of G")
    x = (x_bf16_bits.astype(np.uint32) << 16).view(np.float32).ravel()
    q, S = absmax_quantize(x, G, nthreads)
    q = q.reshape(M, N)
    return q, np.ascontiguousarray(q.T), S.reshape(M, N // G)


def linear_group_quantize(xq: np.ndarray, sx: float, wq: np.ndarray, sw: float, G: int,
                          nthreads: int = 0):
    """FP8 linear layer with a per-group FP8 output -> (y [M, N] float32,
    q [M, N] uint8, S [M, N/G] float32).

    The inputs are quantized per tensor, as the page's mixed-granularity
    scheme has it for linear layers (section 3, "mixed-granularity activation
    quantization", and the section 4 table's row of that name): X = sx
    E4M3(xq) with xq [M, K], W = sw E4M3(wq) with wq [N, K].  y = X W^T,
    rounded once to float32 (the ideal fp32 accumulator).  The output is then
    quantized per 1 x G group along each row, as :func:`absmax_quantize` does
    (section 3, "Triton kernels", linear layer optimisation: the output tile
    is reshaped to (BLOCK_M, BLOCK_N/G, G) and the maximum taken along the
    last axis).

    The sum over K is exact in float64 for K <= 2^17: every E4M3 value is an
    integer multiple of 2^-9 below 2^9, so every product is a multiple of
    2^-18 below 2^18.  sx sw is exact in float64 too; the one float64 rounding
    of (sx sw) times the sum, before the float32 rounding, can only matter
    when it lands exactly on a float32 midpoint.
    """
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    wq = np.ascontiguousarray(wq, dtype=np.uint8)
    M, K = xq.shape
    N, K2 = wq.shape
    if K != K2 or N % G or K > (1 << 17):
        raise ValueError("oracle linear_group_quantize: bad shapes")
    dec = e4m3_decode_all()
    acc = dec[xq] @ dec[wq].T                        # exact (see above)
    y = ((np.float64(np.float32(sx)) * np.float64(np.float32(sw))) * acc).astype(np.float32)
    q, S = absmax_quantize(y, G, nthreads)
    return y, q.reshape(M, N), S.reshape(M, N // G)


def dre_dequantize(q: np.ndarray, S: np.ndarray, k: np.ndarray, G: int,
                   nthreads: int = 0) -> np.ndarray:
    """Inverse of :func:`dre_quantize`: sign(q) (|dec(q)| S)^(1/k) rounded to fp32."""
    lib = _load()
    q = np.ascontiguousarray(q, dtype=np.uint8).ravel()
    S = np.ascontiguousarray(S, dtype=np.float32).ravel()
    k = np.ascontiguousarray(k, dtype=np.float32).ravel()
    n = q.size
    assert S.size == k.size == (n + G - 1) // G
    x = np.zeros(n, dtype=np.float32)
    rc = lib.coat_oracle_dre_dequantize(_ptr(q, ctypes.c_uint8), _ptr(S, ctypes.c_float),
                                        _ptr(k, ctypes.c_float), n, int(G),
                                        _ptr(x, ctypes.c_float), int(nthreads))
    if rc != 0:
        raise ValueError("oracle dre_dequantize: bad arguments")
    return x


def adamw_step(w: np.ndarray, g_bf16_bits: np.ndarray, mq: np.ndarray, vq: np.ndarray,
               meta: np.ndarray, G: int, beta1: float, beta2: float, lr: float, eps: float,
               weight_decay: float, step: int, R: float = R_E4M3_DEFAULT,
               nthreads: int = 0) -> None:
    """One fused AdamW + DRE step, in place on (w, mq, vq, meta).

    ``g_bf16_bits`` holds the bf16 gradient as raw uint16 bits; ``meta`` is
    float32 of shape (num_groups, 4) holding (S_m, k_m, S_v, k_v).
    """
    lib = _load()
    n = w.size
    ng = (n + G - 1) // G
    for a, dt in ((w, np.float32), (g_bf16_bits, np.uint16), (mq, np.uint8), (vq, np.uint8),
                  (meta, np.float32)):
        if a.dtype != dt or not a.flags["C_CONTIGUOUS"]:
            raise TypeError("oracle adamw_step: arrays must be contiguous with the right dtype")
    assert g_bf16_bits.size == n and mq.size == n and vq.size == n and meta.size == 4 * ng
    rc = lib.coat_oracle_adamw_step(_ptr(w, ctypes.c_float), _ptr(g_bf16_bits, ctypes.c_uint16),
                                    _ptr(mq, ctypes.c_uint8), _ptr(vq, ctypes.c_uint8),
                                    _ptr(meta, ctypes.c_float), n, int(G), float(beta1),
                                    float(beta2), float(lr), float(eps), float(weight_decay),
                                    int(step), float(R), int(nthreads))
    if rc != 0:
        raise ValueError("oracle adamw_step: bad arguments")
