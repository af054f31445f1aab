"""SFU throughput on the GB300: exp2 (the fast path's dequantization and
re-encoding use four per parameter) against log2, sqrt and rsqrt.  The step
kernel's SFU floor quoted in the design notes rests on these rates; the test
prints them and checks that exp2 issues at least 1.5 times as fast as log2
(32 against 16 results per SM and clock on this part)."""
import os
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_sfu_rates(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    exe = tmp_path / "sfu_rates"
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                    os.path.join(ROOT, "tests", "native", "sfu_rates.cu"), "-o", str(exe)],
                   check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout
    rates = {k: float(v) for k, v in (ln.split() for ln in out.splitlines() if ln.strip())}
    print(rates)
    assert set(rates) == {"ex2", "lg2", "sqrt", "rsqrt"}
    assert rates["ex2"] >= 1.5 * rates["lg2"]
