"""A recorded hard rounding (tests/golden/hard_rounding_case.txt): the stored
first moment whose dequantized value decides one group's minimum |m_t| at
step 50 of the 4096 x 4096 trajectory, within 3e-7 ulp of an fp32 midpoint.

The oracle rounds it correctly (checked against 50-digit mpmath).  The step
kernel's exact path, run on the host with the same double-float code, must
round it the same way: its double-float value is within its error bound of
the midpoint, so the certain-rounding test sends it to the float64
recomputation.  (Before that test existed the path rounded this value one ulp
off, which moved the group's S_m by 3.96e-6 at step 50 of the 4096 x 4096
trajectory.)
"""
import os

import numpy as np
import pytest

import _exact_path
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


def test_kernel_exact_path_rounds_the_case_correctly(tmp_path):
    exe = _exact_path.build(tmp_path)
    code, S, k, prev, _ = _case()
    got, slow = _exact_path.dequant(exe, [code], [S], [k])
    assert got[0] == abs(prev)
    assert slow[0], "the hard case must be decided by the float64 recomputation"
