"""Host-side check of coat_round.cuh, the certain-rounding test and the
float64 recomputations meant for the exact path's rare hard roundings (CPU
only; the header also compiles for the device)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "coat_fp8_adamw_gb300", "csrc")


def test_round_certain_is_never_wrong(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None:
        pytest.skip("no C++ compiler")
    exe = tmp_path / "round_check"
    subprocess.run([cxx, "-O2", "-std=c++17", "-ffp-contract=off", "-I", CSRC,
                    os.path.join(ROOT, "tests", "native", "round_check.cpp"), "-o", str(exe), "-lm"],
                   check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout
    stats = {k: float(v) for k, v in (kv.split("=") for kv in out.split())}
    print(stats)
    assert stats["random_wrong"] == 0 and stats["near_certain_wrong"] == 0
    assert stats["random_uncertain_frac"] < 1e-4        # about 2 eps / ulp = 2^-15
    assert stats["near_uncertain_frac"] > 0.2           # the uncertain branch is exercised
    assert stats["dequant_diff"] == 0 and stats["k_diff"] == 0


def test_header_compiles_for_the_device(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    src = tmp_path / "use_round.cu"
    src.write_text(
        '#include "coat_round.cuh"\n'
        "__global__ void k(const float* in, float* out, int* flag) {\n"
        "    bool c = false;\n"
        "    out[0] = coat::df::round_certain(coat::df::F2{in[0], in[1]}, 0x1p-40f, c);\n"
        "    flag[0] = c;\n"
        "    out[1] = coat::df::dequant_f64(in[2], in[3], in[4]);\n"
        "    out[2] = coat::df::k_f64(in[5], in[6], 229376.0, 8.0, -125.0, 126.0);\n"
        "}\n")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-std=c++17", "-I", CSRC,
                    "-c", str(src), "-o", str(tmp_path / "use_round.o")], check=True)
