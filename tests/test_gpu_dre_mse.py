"""Quantization error with and without Dynamic Range Expansion, on the GPU
and in the oracle.

The COAT review page's section 4 table credits the expansion with a 1.63x
lower MSE of the stored optimizer states.  This file checks the no-expansion
quantizer (coat_fp8_quantize_absmax) against the oracle, the MSEs of both
storage formats against the oracle's on the same AdamW-like moments, and the
direction of the effect; `bench.py --report dre-mse` measures it at scale.
"""
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import _parity as P
import coat_fp8_adamw_gb300 as coat
import oracle
from coat_fp8_adamw_gb300 import synth

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _built():
    from coat_fp8_adamw_gb300 import _build
    _build.build()
    coat.lib()


def _gpu_absmax(x, G):
    xd = torch.from_numpy(x).cuda()
    q = torch.empty(x.size, dtype=torch.uint8, device="cuda")
    S = torch.empty(coat.num_groups(x.size, G), dtype=torch.float32, device="cuda")
    coat.coat_fp8_quantize_absmax(xd, G, q, S)
    torch.cuda.synchronize()
    return q.cpu().numpy(), S.cpu().numpy()


@pytest.mark.parametrize("G", [1, 2, 4, 8, 16, 32, 64, 128, 256])
def test_absmax_quantizer_matches_oracle(G):
    rng = np.random.default_rng(G + 5)
    n = 4096 * 3 + 77
    x = (rng.standard_normal(n) * 10.0 ** rng.uniform(-12, 4, n)).astype(np.float32)
    x[:G] = 0.0                                   # an all-zero group
    x[-3:] = np.float32(1e-40)                    # subnormal inputs in the ragged group
    q, S = _gpu_absmax(x, G)
    qo, So = oracle.absmax_quantize(x, G)
    assert np.array_equal(S, So), "scales must be bit-identical"
    P.assert_codes_equal(q, qo, f"absmax G={G}")


def _mse(x, back):
    return float(np.mean((back.astype(np.float64) - x.astype(np.float64)) ** 2))


def test_dre_lowers_the_quantization_error_like_the_oracle():
    G, n = 128, 1 << 20
    m, v = synth.adamw_like_moments_np(n, G, 5)
    for name, x in (("m", m), ("v", v)):
        # oracle
        q, S, k = oracle.dre_quantize(x, G)
        mse_dre_o = _mse(x, oracle.dre_dequantize(q, S, k, G))
        q, S = oracle.absmax_quantize(x, G)
        mse_abs_o = _mse(x, oracle.dre_dequantize(q, S, np.ones_like(S), G))
        # GPU, through the C ABI
        xd = torch.from_numpy(x).cuda()
        qd = torch.empty(n, dtype=torch.uint8, device="cuda")
        Sd = torch.empty(n // G, dtype=torch.float32, device="cuda")
        kd = torch.empty(n // G, dtype=torch.float32, device="cuda")
        back = torch.empty(n, dtype=torch.float32, device="cuda")
        coat.coat_dre_quantize(xd, G, qd, Sd, kd)
        coat.coat_dre_dequantize(qd, Sd, kd, G, back)
        mse_dre_g = _mse(x, back.cpu().numpy())
        coat.coat_fp8_quantize_absmax(xd, G, qd, Sd)
        coat.coat_dre_dequantize(qd, Sd, torch.ones_like(Sd), G, back)
        mse_abs_g = _mse(x, back.cpu().numpy())
        print(name, "oracle", mse_abs_o / mse_dre_o, "gpu", mse_abs_g / mse_dre_g)
        assert abs(mse_dre_g / mse_dre_o - 1) < 1e-3
        assert abs(mse_abs_g / mse_abs_o - 1) < 1e-3
        assert mse_abs_o > mse_dre_o and mse_abs_g > mse_dre_g


def test_report_mode_prints_one_json_line():
    r = subprocess.run([sys.executable, "bench.py", "--report", "dre-mse", "--params", str(1 << 22)],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for name in ("m", "v"):
        assert line["moments"][name]["no_dre_over_dre"] > 1.0
    for kern in ("dre_quantize", "fp8_quantize_absmax", "dre_dequantize"):
        assert line["kernels"][kern]["achieved_gbs"] > 0
