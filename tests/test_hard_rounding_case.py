"""A recorded hard rounding (tests/golden/hard_rounding_case.txt): the stored
first moment whose dequantized value decides one group's minimum |m_t| at
step 50 of the 4096 x 4096 trajectory, within 3e-7 ulp of an fp32 midpoint.

The oracle rounds it correctly (checked against 50-digit mpmath).  The step
kernel's exact path, run on the host with the same double-float code, rounds
it one ulp off: the known gap that the teacher-forced GPU check along that
trajectory reports, kept here as an expected failure until the exact path
rounds such cases with certainty.
"""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CASE = os.path.join(ROOT, "tests", "golden", "hard_rounding_case.txt")


def _case():
    with open(CASE) as fh:
        line = [ln for ln in fh if not ln.startswith("#")][0]
    code, s, k, prev, g = (int(x) for x in line.split())
    return (code, np.uint32(s).view(np.float32), np.uint32(k).view(np.float32),
            np.uint32(prev).view(np.float32), np.uint32(g).view(np.float32))


def test_oracle_value_is_the_correct_rounding():
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 50
    code, S, k, prev, _ = _case()
    assert oracle.dre_dequantize(np.array([code], np.uint8), np.array([S]), np.array([k]), 1)[0] == prev
    x = mpmath.power(mpmath.mpf(float(abs(oracle.e4m3_decode_all()[code]))) * mpmath.mpf(float(S)),
                     1 / mpmath.mpf(float(k)))
    lo, hi = np.nextafter(prev, np.float32(0)), np.nextafter(prev, np.float32(np.inf))
    # prev is the nearest float, and the exact value sits close to a midpoint
    assert abs(x - mpmath.mpf(float(prev))) < abs(x - mpmath.mpf(float(lo)))
    assert abs(x - mpmath.mpf(float(prev))) < abs(x - mpmath.mpf(float(hi)))
    ulp = mpmath.mpf(float(hi)) - mpmath.mpf(float(prev))
    assert abs(abs(x - mpmath.mpf(float(prev))) / ulp - mpmath.mpf(0.5)) < 1e-6


@pytest.mark.xfail(strict=False, reason=(
    "known gap: the exact path rounds a double-float value accurate to about "
    "2^-44 once, and this value lies within 3e-7 ulp of an fp32 midpoint"))
def test_kernel_exact_path_rounds_the_case_correctly(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    exe = tmp_path / "exact_path"
    subprocess.run([cxx, "-O2", "-std=c++17", "-ffp-contract=off", "-I",
                    os.path.join(ROOT, "coat_fp8_adamw_gb300", "csrc"),
                    os.path.join(ROOT, "tests", "native", "exact_path.cpp"), "-o", str(exe)],
                   check=True)
    code, S, k, prev, _ = _case()
    out = subprocess.run([str(exe), str(code), str(int(S.view(np.uint32))), str(int(k.view(np.uint32)))],
                         capture_output=True, text=True, check=True).stdout
    assert np.uint32(int(out)).view(np.float32) == prev
