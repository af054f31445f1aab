"""The kernels' constant table (coat_tables.inc) is the committed output of
gen_tables.py and agrees with the oracle's E4M3 decoding (CPU only)."""
import math
import os
import re
import struct
import subprocess
import sys

import numpy as np

import oracle

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "coat_fp8_adamw_gb300", "csrc")


def _tables():
    src = open(os.path.join(CSRC, "coat_tables.inc")).read()
    out = {}
    for name, body in re.findall(r"(kLog2Frac448\w+)\[128\] = \{(.*?)\};", src, flags=re.S):
        bits = [int(t.strip().rstrip("u"), 16) for t in body.split(",") if t.strip()]
        out[name] = np.array([struct.unpack("<f", struct.pack("<I", b))[0] for b in bits])
    return out


def test_committed_table_is_generator_output():
    fresh = subprocess.run([sys.executable, "gen_tables.py"], cwd=CSRC, capture_output=True,
                           text=True, check=True).stdout
    assert fresh == open(os.path.join(CSRC, "coat_tables.inc")).read()


def test_table_matches_oracle_decode():
    t = _tables()
    hi, lo = t["kLog2Frac448Hi"], t["kLog2Frac448Lo"]
    assert hi.size == lo.size == 128
    vals = oracle.e4m3_decode_all()
    for c in range(1, 127):
        want = math.log2(vals[c] / 448.0)
        assert abs(float(hi[c]) + float(lo[c]) - want) <= 1e-13 * max(1.0, abs(want)), c
        assert abs(float(hi[c]) - want) <= 2.0 ** -24 * abs(want) + 1e-30, c
    assert hi[0] < -1e29 and hi[0x7E] == 0.0 and hi[0x7F] == 0.0


def _gen_tables_module():
    import importlib.util
    spec = importlib.util.spec_from_file_location("gen_tables", os.path.join(CSRC, "gen_tables.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_generator_fp32_rounding_matches_numpy():
    """The generator's exact fp32 rounding (used to repeat the kernels' FMA
    chain for the log2 reciprocals) rounds like numpy's float64 -> float32
    conversion, ties to even included."""
    from fractions import Fraction
    g = _gen_tables_module()
    rng = np.random.default_rng(7)
    vals = list(rng.standard_normal(3000) * np.exp2(rng.integers(-60, 60, 3000)))
    # exact ties: a float32 plus half its spacing, both parities
    for f in rng.standard_normal(500).astype(np.float32):
        up = np.nextafter(f, np.float32(np.inf), dtype=np.float32)
        vals.append((float(f) + float(up)) / 2.0)
    for v in vals:
        want = float(np.float32(v))
        assert float(g.rn32(Fraction(v))) == want, v


def test_log2_reciprocals_keep_the_reduction_exact():
    """Every interval's reciprocal, as the generator derives it from the
    kernels' quartic, keeps |u r_j - 1| below 2^-8 over the interval."""
    from fractions import Fraction
    g = _gen_tables_module()
    poly = g.recip_poly()
    for j in range(256):
        M = g.log_reduction_numerator(j, poly)
        r = Fraction(M, 512)
        for u in (1 + Fraction(j, 256), 1 + Fraction(j + 1, 256) - Fraction(1, 1 << 23)):
            assert abs(u * r - 1) < Fraction(1, 256)
