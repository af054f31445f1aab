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
