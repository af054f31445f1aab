"""Python binding of libcoat_gb300 (the C ABI declared in include/coat.h).

This module only marshals arguments: it checks tensor dtypes, devices and
shapes, passes raw device pointers and the current CUDA stream through
ctypes, and turns a non-zero status into :class:`CoatError`.  Every step of
the optimizer runs in the library's CUDA kernels.  There is no CPU or PyTorch
fallback: if the shared library has not been built, every call raises.

Build it with ``python -c "import __graft_entry__ as g; g.build()"`` (or
``python coat_fp8_adamw_gb300/_build.py``).
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

from . import _build

__all__ = ["CoatError", "coat_fp8_adamw_step", "coat_fp8_adamw_step_host",
           "coat_fp8_adamw_step_host_workspace_bytes", "coat_fp8_adamw_step_host_static",
           "coat_dre_quantize", "coat_fp8_quantize_absmax", "coat_act_quantize_fp8",
           "coat_fp8_linear_group_quantize",
           "coat_dre_dequantize", "coat_exact_recompute_counts", "coat_kernel_wait_timeouts",
           "coat_status_string",
           "coat_r_e4m3", "coat_version", "lib",
           "lib_path", "num_groups", "bytes_per_param", "STATUS",
           "STATIC_SCRATCH_BYTES", "MAX_N"]

STATUS = {0: "COAT_OK", 1: "COAT_ERR_INVALID_ARG", 2: "COAT_ERR_MISALIGNED",
          3: "COAT_ERR_UNSUPPORTED_G", 4: "COAT_ERR_CUDA", 5: "COAT_ERR_NOT_DEVICE",
          6: "COAT_ERR_SCRATCH_LIMIT"}

#: COAT_STATIC_SCRATCH_BYTES of include/coat.h
STATIC_SCRATCH_BYTES = 16 << 20

#: COAT_MAX_N of include/coat.h: the largest element count any entry point accepts
MAX_N = 1 << 40

#: symbols the shared library must export (one per declaration in include/coat.h)
EXPORTS = ("coat_fp8_adamw_step", "coat_fp8_adamw_step_host",
           "coat_fp8_adamw_step_host_workspace_bytes", "coat_fp8_adamw_step_host_static",
           "coat_dre_quantize", "coat_fp8_quantize_absmax", "coat_act_quantize_fp8",
           "coat_fp8_linear_group_quantize",
           "coat_dre_dequantize", "coat_exact_recompute_counts", "coat_kernel_wait_timeouts",
           "coat_status_string",
           "coat_r_e4m3", "coat_version")

_lock = threading.Lock()
_lib = None


class CoatError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = coat_status_string(status) if _lib is not None else STATUS.get(status, "?")
        super().__init__(f"{where}: {STATUS.get(status, status)} ({msg})")


def lib_path() -> str:
    return _build.lib_path()


def lib() -> ctypes.CDLL:
    """The loaded library.  Raises if it has not been built: no fallback exists."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = lib_path()
        if not os.path.exists(path):
            raise RuntimeError(
                f"libcoat_gb300 is not built ({path} missing); run "
                "`python -c 'import __graft_entry__ as g; g.build()'` first")
        L = ctypes.CDLL(path)
        vp, i64, i32, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float
        L.coat_fp8_adamw_step.argtypes = [vp, vp, vp, vp, vp, i64, i32, f32, f32, f32, f32, f32,
                                          i64, vp]
        L.coat_fp8_adamw_step.restype = ctypes.c_int
        L.coat_fp8_adamw_step_host.argtypes = [vp, vp, vp, vp, vp, i64, i32, f32, f32, f32, f32,
                                               f32, i64, vp, ctypes.c_size_t, vp]
        L.coat_fp8_adamw_step_host.restype = ctypes.c_int
        L.coat_fp8_adamw_step_host_workspace_bytes.argtypes = [i64, i32]
        L.coat_fp8_adamw_step_host_workspace_bytes.restype = ctypes.c_size_t
        L.coat_fp8_adamw_step_host_static.argtypes = [vp, vp, vp, vp, vp, i64, i32, f32, f32, f32,
                                                      f32, f32, i64, i64, vp]
        L.coat_fp8_adamw_step_host_static.restype = ctypes.c_int
        L.coat_dre_quantize.argtypes = [vp, i64, i32, vp, vp, vp, vp]
        L.coat_dre_quantize.restype = ctypes.c_int
        L.coat_fp8_quantize_absmax.argtypes = [vp, i64, i32, vp, vp, vp]
        L.coat_fp8_quantize_absmax.restype = ctypes.c_int
        L.coat_act_quantize_fp8.argtypes = [vp, i64, i64, i32, vp, vp, vp, vp]
        L.coat_act_quantize_fp8.restype = ctypes.c_int
        L.coat_fp8_linear_group_quantize.argtypes = [vp, f32, vp, f32, i64, i64, i64, i32, vp, vp,
                                                     vp, vp]
        L.coat_fp8_linear_group_quantize.restype = ctypes.c_int
        L.coat_dre_dequantize.argtypes = [vp, vp, vp, i64, i32, vp, vp]
        L.coat_dre_dequantize.restype = ctypes.c_int
        L.coat_exact_recompute_counts.argtypes = [vp, i32]
        L.coat_exact_recompute_counts.restype = ctypes.c_int
        L.coat_kernel_wait_timeouts.argtypes = [vp, i32]
        L.coat_kernel_wait_timeouts.restype = ctypes.c_int
        L.coat_status_string.argtypes = [ctypes.c_int]
        L.coat_status_string.restype = ctypes.c_char_p
        L.coat_r_e4m3.argtypes = []
        L.coat_r_e4m3.restype = ctypes.c_double
        L.coat_version.argtypes = []
        L.coat_version.restype = ctypes.c_int32
        _lib = L
        return L


def coat_exact_recompute_counts(reset: bool = False, device=None) -> tuple:
    """(dequantized moments, exponents k) that the step's exact path recomputed
    in float64 on ``device`` (default: the current one) since load or the last
    reset.  Synchronizes with that device."""
    import torch
    out = (ctypes.c_uint64 * 2)()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    with torch.cuda.device(dev):
        st = lib().coat_exact_recompute_counts(ctypes.cast(out, ctypes.c_void_p), int(bool(reset)))
    if st != 0:
        raise CoatError(st, "coat_exact_recompute_counts")
    return int(out[0]), int(out[1])


def coat_kernel_wait_timeouts(reset: bool = False, device=None) -> int:
    """Bounded waits inside the library's pipelined kernels that gave up on
    ``device`` (default: the current one) since load or the last reset; a
    non-zero count means a launch returned unfinished.  Synchronizes."""
    import torch
    out = ctypes.c_uint64(0)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    with torch.cuda.device(dev):
        st = lib().coat_kernel_wait_timeouts(ctypes.byref(out), int(bool(reset)))
    if st != 0:
        raise CoatError(st, "coat_kernel_wait_timeouts")
    return int(out.value)


def coat_status_string(status: int) -> str:
    return lib().coat_status_string(int(status)).decode()


def coat_r_e4m3() -> float:
    return float(lib().coat_r_e4m3())


def coat_version() -> int:
    return int(lib().coat_version())


def num_groups(n: int, G: int) -> int:
    return (n + G - 1) // G


def bytes_per_param(G: int) -> float:
    """Algorithmic HBM traffic of one step per parameter (read + write).

    w fp32 read+write 8 B, g bf16 read 2 B, m and v codes read+write 4 B, and
    the 16-byte (S_m, k_m, S_v, k_v) record of each group read+write 32/G B.
    """
    return 14.0 + 32.0 / G


# ---------------------------------------------------------------------------
# torch-tensor front end
# ---------------------------------------------------------------------------

def _stream_ptr(stream, device=None) -> Optional[int]:
    """The stream handle to pass: ``stream``, or the current torch stream of
    ``device`` (the device the tensors live on; the call runs with it current)."""
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _check(t, dtype, numel: int, name: str, device=None):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must have dtype {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.numel() != numel:
        raise ValueError(f"{name} must have {numel} elements, got {t.numel()}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    return t.data_ptr()


def coat_fp8_adamw_step(w, g, m_q, v_q, meta, G: int, beta1: float, beta2: float, lr: float,
                        eps: float, weight_decay: float, step: int, stream=None) -> None:
    """One fused FP8 AdamW + DRE step, in place on w, m_q, v_q and meta.

    w fp32 [n]; g bf16 [n]; m_q, v_q uint8 [n]; meta fp32 [ceil(n/G), 4]
    holding (S_m, k_m, S_v, k_v) per group.  Runs on ``stream`` (default: the
    current torch stream) and returns without synchronizing.
    """
    import torch
    n = w.numel()
    dev = w.device
    pw = _check(w, torch.float32, n, "w")
    pg = _check(g, torch.bfloat16, n, "g", dev)
    pm = _check(m_q, torch.uint8, n, "m_q", dev)
    pv = _check(v_q, torch.uint8, n, "v_q", dev)
    pmeta = _check(meta, torch.float32, 4 * num_groups(n, G), "meta", dev)
    with torch.cuda.device(dev):
        st = lib().coat_fp8_adamw_step(pw, pg, pm, pv, pmeta, n, int(G), float(beta1), float(beta2),
                                       float(lr), float(eps), float(weight_decay), int(step),
                                       _stream_ptr(stream))
    if st != 0:
        raise CoatError(st, "coat_fp8_adamw_step")


def coat_fp8_adamw_step_host_workspace_bytes(chunk_params: int, G: int) -> int:
    return int(lib().coat_fp8_adamw_step_host_workspace_bytes(int(chunk_params), int(G)))


def _check_host(t, dtype, numel: int, name: str):
    import torch
    if not isinstance(t, torch.Tensor) or t.dtype != dtype or t.is_cuda:
        raise TypeError(f"{name} must be a CPU tensor of dtype {dtype}")
    if not t.is_contiguous() or t.numel() != numel:
        raise ValueError(f"{name} must be contiguous with {numel} elements")
    return t.data_ptr()


def coat_fp8_adamw_step_host(w, g, m_q, v_q, meta, G: int, beta1: float, beta2: float, lr: float,
                             eps: float, weight_decay: float, step: int, workspace,
                             stream=None) -> None:
    """The step on host (ideally pinned) CPU tensors, streamed through the
    device tensor ``workspace`` (uint8, see coat_fp8_adamw_step_host_workspace_bytes).
    Returns when the host tensors hold the result."""
    import torch
    n = w.numel()
    pw = _check_host(w, torch.float32, n, "w")
    pg = _check_host(g, torch.bfloat16, n, "g")
    pm = _check_host(m_q, torch.uint8, n, "m_q")
    pv = _check_host(v_q, torch.uint8, n, "v_q")
    pmeta = _check_host(meta, torch.float32, 4 * num_groups(n, G), "meta")
    if not (isinstance(workspace, torch.Tensor) and workspace.is_cuda and workspace.is_contiguous()):
        raise TypeError("workspace must be a contiguous CUDA tensor")
    with torch.cuda.device(workspace.device):
        st = lib().coat_fp8_adamw_step_host(pw, pg, pm, pv, pmeta, n, int(G), float(beta1),
                                            float(beta2), float(lr), float(eps),
                                            float(weight_decay), int(step), workspace.data_ptr(),
                                            workspace.numel() * workspace.element_size(),
                                            _stream_ptr(stream))
    if st != 0:
        raise CoatError(st, "coat_fp8_adamw_step_host")


def coat_fp8_adamw_step_host_static(w, g, m_q, v_q, meta, G: int, beta1: float, beta2: float,
                                    lr: float, eps: float, weight_decay: float, step: int,
                                    chunk_params: int = 0, stream=None) -> None:
    """The step on host CPU tensors through the library's fixed device scratch
    (COAT_STATIC_SCRATCH_BYTES): no device allocation, for callers that cannot
    allocate.  Calls on one device must not overlap in time.  Returns when the
    host tensors hold the result."""
    import torch
    n = w.numel()
    pw = _check_host(w, torch.float32, n, "w")
    pg = _check_host(g, torch.bfloat16, n, "g")
    pm = _check_host(m_q, torch.uint8, n, "m_q")
    pv = _check_host(v_q, torch.uint8, n, "v_q")
    pmeta = _check_host(meta, torch.float32, 4 * num_groups(n, G), "meta")
    # the call runs on the stream's device (the current one when no stream is given)
    dev = stream.device if isinstance(stream, torch.cuda.Stream) else torch.device(
        "cuda", torch.cuda.current_device())
    with torch.cuda.device(dev):
        st = lib().coat_fp8_adamw_step_host_static(pw, pg, pm, pv, pmeta, n, int(G), float(beta1),
                                                   float(beta2), float(lr), float(eps),
                                                   float(weight_decay), int(step),
                                                   int(chunk_params), _stream_ptr(stream, dev))
    if st != 0:
        raise CoatError(st, "coat_fp8_adamw_step_host_static")


def coat_dre_quantize(x, G: int, q, scale, k, stream=None) -> None:
    """DRE + E4M3 quantization: x fp32 [n] -> q uint8 [n], scale/k fp32 [ceil(n/G)]."""
    import torch
    n = x.numel()
    ng = num_groups(n, G)
    px = _check(x, torch.float32, n, "x")
    pq = _check(q, torch.uint8, n, "q", x.device)
    ps = _check(scale, torch.float32, ng, "scale", x.device)
    pk = _check(k, torch.float32, ng, "k", x.device)
    with torch.cuda.device(x.device):
        st = lib().coat_dre_quantize(px, n, int(G), pq, ps, pk, _stream_ptr(stream))
    if st != 0:
        raise CoatError(st, "coat_dre_quantize")


def coat_fp8_quantize_absmax(x, G: int, q, scale, stream=None) -> None:
    """Per-group FP8 without the expansion: x fp32 [n] -> q uint8 [n], scale fp32 [ceil(n/G)]
    (scale = max|x| / 448; decode with coat_dre_dequantize and k = 1)."""
    import torch
    n = x.numel()
    ng = num_groups(n, G)
    px = _check(x, torch.float32, n, "x")
    pq = _check(q, torch.uint8, n, "q", x.device)
    ps = _check(scale, torch.float32, ng, "scale", x.device)
    with torch.cuda.device(x.device):
        st = lib().coat_fp8_quantize_absmax(px, n, int(G), pq, ps, _stream_ptr(stream))
    if st != 0:
        raise CoatError(st, "coat_fp8_quantize_absmax")


def coat_act_quantize_fp8(x, G: int, q, scale, qt=None, stream=None) -> None:
    """Per-group (1 x G) FP8 quantization of a bf16 activation x [M, N]:
    q uint8 [M, N], scale fp32 [M, N/G], and optionally qt uint8 [N, M] (the codes transposed)."""
    import torch
    if x.dim() != 2:
        raise ValueError("x must be a 2-D [M, N] tensor")
    M, N = x.shape
    px = _check(x, torch.bfloat16, M * N, "x")
    pq = _check(q, torch.uint8, M * N, "q", x.device)
    ps = _check(scale, torch.float32, (M * N) // G if G > 0 else 0, "scale", x.device)
    pqt = _check(qt, torch.uint8, M * N, "qt", x.device) if qt is not None else None
    with torch.cuda.device(x.device):
        st = lib().coat_act_quantize_fp8(px, M, N, int(G), pq, pqt, ps, _stream_ptr(stream))
    if st != 0:
        raise CoatError(st, "coat_act_quantize_fp8")


def coat_fp8_linear_group_quantize(xq, sx: float, wq, sw: float, G: int, q, scale, y=None,
                                   stream=None) -> None:
    """FP8 linear layer with a per-group FP8 output: y = (sx E4M3(xq)) (sw E4M3(wq))^T
    for xq uint8 [M, K] and wq uint8 [N, K], quantized per 1 x G group of each row
    into q uint8 [M, N] and scale fp32 [M, N/G]; y fp32 [M, N] is written when given."""
    import torch
    if xq.dim() != 2 or wq.dim() != 2 or xq.shape[1] != wq.shape[1]:
        raise ValueError("xq [M, K] and wq [N, K] must be 2-D with the same K")
    (M, K), N = xq.shape, wq.shape[0]
    px = _check(xq, torch.uint8, M * K, "xq")
    pw = _check(wq, torch.uint8, N * K, "wq", xq.device)
    pq = _check(q, torch.uint8, M * N, "q", xq.device)
    ps = _check(scale, torch.float32, (M * N) // G if G > 0 else 0, "scale", xq.device)
    py = _check(y, torch.float32, M * N, "y", xq.device) if y is not None else None
    with torch.cuda.device(xq.device):
        st = lib().coat_fp8_linear_group_quantize(px, float(sx), pw, float(sw), M, N, K, int(G),
                                                  pq, ps, py, _stream_ptr(stream))
    if st != 0:
        raise CoatError(st, "coat_fp8_linear_group_quantize")


def coat_dre_dequantize(q, scale, k, G: int, x, stream=None) -> None:
    """Inverse of :func:`coat_dre_quantize`: x = sign(q)(|E4M3(q)| scale)^(1/k)."""
    import torch
    n = q.numel()
    ng = num_groups(n, G)
    pq = _check(q, torch.uint8, n, "q")
    ps = _check(scale, torch.float32, ng, "scale", q.device)
    pk = _check(k, torch.float32, ng, "k", q.device)
    px = _check(x, torch.float32, n, "x", q.device)
    with torch.cuda.device(q.device):
        st = lib().coat_dre_dequantize(pq, ps, pk, n, int(G), px, _stream_ptr(stream))
    if st != 0:
        raise CoatError(st, "coat_dre_dequantize")
