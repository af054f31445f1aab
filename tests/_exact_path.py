"""Build and drive tests/native/exact_path.cpp: the step kernel's exact path
(certain rounding with a float64 fallback) compiled for the host."""
import os
import shutil
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "coat_fp8_adamw_gb300", "csrc")


def build(tmp_dir) -> str:
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    exe = os.path.join(str(tmp_dir), "exact_path")
    subprocess.run([cxx, "-O2", "-std=c++17", "-ffp-contract=off", "-I", CSRC,
                    os.path.join(ROOT, "tests", "native", "exact_path.cpp"), "-o", exe, "-lm"],
                   check=True)
    return exe


def _run(exe, lines):
    out = subprocess.run([exe], input="\n".join(lines) + "\n", capture_output=True, text=True,
                         check=True).stdout.split()
    vals = np.array([int(x) for x in out[0::2]], dtype=np.uint32).view(np.float32)
    slow = np.array([int(x) for x in out[1::2]], dtype=bool)
    return vals, slow


def dequant(exe, codes, S, k):
    """Dequantized magnitudes (|E4M3(code)| S)^(1/k) and the float64-path flags."""
    S = np.asarray(S, np.float32)
    k = np.asarray(k, np.float32)
    lines = [f"d {int(c)} {int(s)} {int(kk)}"
             for c, s, kk in zip(codes, S.view(np.uint32), k.view(np.uint32))]
    return _run(exe, lines)


def kexp(exe, mx, mn):
    """Group exponents k for extremes mx >= mn > 0 and the float64-path flags."""
    mx = np.asarray(mx, np.float32)
    mn = np.asarray(mn, np.float32)
    lines = [f"k {int(a)} {int(b)}" for a, b in zip(mx.view(np.uint32), mn.view(np.uint32))]
    return _run(exe, lines)
