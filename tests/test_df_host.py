"""Host-side check of the kernels' double-float toolkit (CPU only).

coat_df.cuh is built only from IEEE add / multiply / fma / divide, so the
same code compiled for the host gives the results the device gets.  The
harness in tests/native/df_check.cpp compares it with float64 libm and long
double, checks the log2 reduction exhaustively, and measures the margin of the
error bounds that the certain-rounding test of coat_round.cuh relies on.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_double_float_toolkit_accuracy(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    exe = tmp_path / "df_check"
    subprocess.run([cxx, "-O2", "-std=c++17", "-ffp-contract=off",
                    "-I", os.path.join(ROOT, "coat_fp8_adamw_gb300", "csrc"),
                    os.path.join(ROOT, "tests", "native", "df_check.cpp"), "-o", str(exe), "-lm"],
                   check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout
    stats = dict(kv.split("=") for kv in out.split())
    stats = {k: float(v) for k, v in stats.items()}
    print(stats)
    assert stats["log2_max_abs"] < 2.0 ** -40          # |log2 x| <= 149: ~2^-48 relative
    assert stats["log2_max_abs_near1"] < 2.0 ** -46
    # the reduction u r_j - 1 is exact for every significand, |t| < 2^-8.38,
    # and log2 of every significand is within 2^-47 (the table matches r_j)
    assert stats["reduce_inexact"] == 0
    assert stats["reduce_max"] < 2.0 ** -8.38
    assert stats["log2_sig_max_abs"] < 2.0 ** -47
    # log2 within its stated bound 2^-46 + 2^-47 |log2 x|, with room to spare
    assert stats["log2_bound_ratio"] < 0.75
    # the certain-rounding test's error bounds keep a margin of at least 2
    # over the largest errors of the values they bound
    assert 0.0 < stats["dequant_bound_ratio"] < 0.5
    assert 0.0 < stats["k_bound_ratio"] < 0.5
    # x 2^n is the correctly rounded product for every exponent, subnormal
    # results and the clamped range included
    assert stats["scale2_miss"] == 0
    assert stats["exp2_miss_frac"] < 1e-5              # correctly rounded except near ties
    assert stats["exp2_max_rel"] <= 2.0 ** -24 * 1.0001
    assert stats["div_miss_frac"] < 1e-5
    assert stats["dot_miss_frac"] < 1e-5
