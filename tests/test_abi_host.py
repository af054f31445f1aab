"""The C-ABI library loads, exports every declared symbol, and validates
arguments on the host (CPU only: no call here reaches a kernel)."""
import os
import re

import pytest

import coat_fp8_adamw_gb300 as coat
from coat_fp8_adamw_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    _build.build()
    return coat.lib()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "coat.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(coat_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(L):
    declared = _declared_functions()
    assert set(declared) == set(coat.EXPORTS)
    for name in declared:
        assert hasattr(L, name), name


def test_constants(L):
    assert coat.coat_r_e4m3() == 448.0 * 2 ** 9
    assert coat.coat_version() >= 100
    for s, name in coat.STATUS.items():
        assert coat.coat_status_string(s)
    assert coat.coat_status_string(99) == "unknown status"


A = 1 << 20  # a 16-byte aligned fake address: validation must reject before any access


def _step(L, w=A, g=A + 0x100000, mq=A + 0x200000, vq=A + 0x300000, meta=A + 0x400000, n=256,
          G=128, b1=0.9, b2=0.95, lr=1e-4, eps=1e-8, wd=0.1, step=1):
    return L.coat_fp8_adamw_step(w, g, mq, vq, meta, n, G, b1, b2, lr, eps, wd, step, None)


def test_step_validation(L):
    assert _step(L, w=0) == 1
    assert _step(L, n=0) == 1
    assert _step(L, step=0) == 1
    for G in (0, 3, 96, 512, -4):
        assert _step(L, G=G) == 3
    assert _step(L, w=A + 4) == 2
    assert _step(L, meta=A + 0x400008) == 2
    assert _step(L, b1=1.0) == 1
    assert _step(L, b2=-0.1) == 1
    assert _step(L, lr=float("nan")) == 1
    assert _step(L, eps=0.0) == 1
    assert _step(L, wd=-1.0) == 1
    assert _step(L, g=A + 16) == 1              # gradient overlaps the weights
    assert _step(L, vq=A + 0x200000 + 128) == 1  # codes overlap
    # a well-formed call on memory that is not device memory is refused
    assert _step(L) == 5


def test_header_constants_match_the_binding():
    src = open(os.path.join(ROOT, "include", "coat.h")).read()
    assert re.search(r"#define COAT_MAX_N \(\(int64_t\)1 << 40\)", src)
    assert re.search(r"#define COAT_STATIC_SCRATCH_BYTES \(\(size_t\)16 << 20\)", src)
    assert coat.MAX_N == 1 << 40 and coat.STATIC_SCRATCH_BYTES == 16 << 20


def test_sizes_beyond_the_limit_are_refused(L):
    big = coat.MAX_N + 1
    assert _step(L, n=big) == 1
    assert _static(L, n=big) == 1
    assert L.coat_dre_quantize(A, big, 16, A + 4096, A + 8192, A + 12288, None) == 1
    assert L.coat_fp8_quantize_absmax(A, big, 16, A + 4096, A + 8192, None) == 1
    assert L.coat_dre_dequantize(A, A + 4096, A + 8192, big, 16, A + 12288, None) == 1
    assert L.coat_fp8_adamw_step_host(A, A + 0x100000, A + 0x200000, A + 0x300000, A + 0x400000,
                                      big, 128, 0.9, 0.95, 1e-4, 1e-8, 0.1, 1, A + 0x500000,
                                      1 << 20, None) == 1


def test_codec_validation(L):
    assert L.coat_dre_quantize(0, 16, 16, A, A + 4096, A + 8192, None) == 1
    assert L.coat_dre_quantize(A, 16, 7, A + 4096, A + 8192, A + 12288, None) == 3
    assert L.coat_dre_quantize(A + 8, 16, 16, A + 4096, A + 8192, A + 12288, None) == 2
    assert L.coat_dre_quantize(A, 64, 16, A + 16, A + 8192, A + 12288, None) == 1
    assert L.coat_dre_quantize(A, 64, 16, A + 4096, A + 8192, A + 12288, None) == 5
    assert L.coat_dre_dequantize(A, A + 4096, A + 8192, 0, 16, A + 12288, None) == 1
    assert L.coat_dre_dequantize(A, A + 4096, A + 8192, 64, 16, A + 12288, None) == 5


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(coat, "_lib", None)
    monkeypatch.setattr(coat._build, "lib_path", lambda: str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        coat.lib()


def _static(L, chunk=0, w=A, g=A + 0x100000, mq=A + 0x200000, vq=A + 0x300000, meta=A + 0x400000,
            n=256, G=128, step=1):
    return L.coat_fp8_adamw_step_host_static(w, g, mq, vq, meta, n, G, 0.9, 0.95, 1e-4, 1e-8, 0.1,
                                             step, chunk, None)


def test_static_scratch_limits(L):
    """Requests beyond the static scratch are refused before any pointer is used."""
    assert _static(L, chunk=-1) == 1
    assert _static(L, n=0) == 1
    assert _static(L, G=3) == 3
    assert _static(L, chunk=coat.STATIC_SCRATCH_BYTES + 1) == 6
    assert _static(L, chunk=1 << 62) == 6
    # one chunk of c parameters needs 8c bytes plus 16 per group, each part rounded to 256
    assert _static(L, chunk=2_100_000) == 6
    assert _static(L, G=1, chunk=700_000) == 6
    assert coat.coat_status_string(6) == "request exceeds the library's static scratch"


def test_absmax_quantizer_validation(L):
    assert L.coat_fp8_quantize_absmax(0, 16, 16, A, A + 4096, None) == 1
    assert L.coat_fp8_quantize_absmax(A, 0, 16, A + 4096, A + 8192, None) == 1
    assert L.coat_fp8_quantize_absmax(A, 16, 12, A + 4096, A + 8192, None) == 3
    assert L.coat_fp8_quantize_absmax(A + 4, 16, 16, A + 4096, A + 8192, None) == 2
    assert L.coat_fp8_quantize_absmax(A, 64, 16, A + 16, A + 8192, None) == 1   # x overlaps q
    assert L.coat_fp8_quantize_absmax(A, 64, 16, A + 4096, A + 8192, None) == 5


def _lin(L, xq=A, sx=1.0, wq=A + 0x100000, sw=1.0, M=128, N=128, K=64, G=16, q=A + 0x200000,
         S=A + 0x300000, y=None):
    return L.coat_fp8_linear_group_quantize(xq, sx, wq, sw, M, N, K, G, q, S, y, None)


def test_linear_validation(L):
    assert _lin(L, xq=0) == 1 and _lin(L, M=0) == 1 and _lin(L, K=0) == 1
    assert _lin(L, sx=0.0) == 1 and _lin(L, sw=-1.0) == 1 and _lin(L, sx=float("inf")) == 1
    assert _lin(L, G=4) == 3 and _lin(L, G=256) == 3 and _lin(L, G=24) == 3
    assert _lin(L, N=120) == 1 and _lin(L, N=48, G=32) == 1 and _lin(L, K=40) == 1
    assert _lin(L, M=1 << 31) == 1                            # TMA coordinates are 32-bit
    assert _lin(L, q=A + 0x200008) == 2 and _lin(L, y=A + 0x400004) == 2
    assert _lin(L, q=A + 0x100000) == 1                      # q overlaps wq
    assert _lin(L, y=A + 0x300000) == 1                      # y overlaps the scales
    assert _lin(L) == 5 and _lin(L, y=A + 0x400000) == 5      # not device memory here
    assert _lin(L, M=1, N=16, K=16) == 5                      # ragged sizes pass validation
    assert L.coat_kernel_wait_timeouts(None, 0) == 1
