"""GPU parity of the standalone DRE quantizer / dequantizer against the oracle."""
import math

import numpy as np
import pytest
import torch

import _parity as P
import coat_fp8_adamw_gb300 as coat
import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from coat_fp8_adamw_gb300 import _build
    _build.build()
    coat.lib()


def _groups(G, count, seed):
    rng = np.random.default_rng(seed)
    parts = []
    for i in range(count):
        kind = i % 6
        s = 10.0 ** rng.uniform(-12, 2)
        if kind == 0:
            x = rng.standard_normal(G) * s
        elif kind == 1:
            x = rng.standard_normal(G) ** 2 * s
        elif kind == 2:
            x = np.exp(rng.uniform(-30, 0, G)) * s * np.sign(rng.standard_normal(G))
        elif kind == 3:
            x = np.zeros(G); x[rng.integers(G)] = s          # single non-zero (or all-zero when G==1)
        elif kind == 4:
            x = (1 + 0.01 * rng.random(G)) * s               # near-equal: k cap
        else:
            x = rng.standard_normal(G) * 1e-36               # tiny: S guard
        parts.append(x)
    return np.concatenate(parts).astype(np.float32)


def gpu_quantize(x, G):
    n = x.size
    ng = (n + G - 1) // G
    xd = torch.from_numpy(x).cuda()
    q = torch.empty(n, dtype=torch.uint8, device="cuda")
    S = torch.empty(ng, device="cuda")
    k = torch.empty(ng, device="cuda")
    coat.coat_dre_quantize(xd, G, q, S, k)
    torch.cuda.synchronize()
    return q.cpu().numpy(), S.cpu().numpy(), k.cpu().numpy()


def gpu_dequantize(q, S, k, G):
    qd = torch.from_numpy(q).cuda()
    x = torch.empty(q.size, device="cuda")
    coat.coat_dre_dequantize(qd, torch.from_numpy(S).cuda(), torch.from_numpy(k).cuda(), G, x)
    torch.cuda.synchronize()
    return x.cpu().numpy()


@pytest.mark.parametrize("G", [1, 2, 4, 8, 16, 32, 64, 128, 256])
def test_quantize_matches_oracle(G):
    x = _groups(G, max(64, 8192 // G), seed=G)
    x = np.concatenate([x, x[:G // 2 + 3]])                 # ragged tail
    qg, Sg, kg = gpu_quantize(x, G)
    qo, So, ko = oracle.dre_quantize(x, G)
    st = P.compare_codes(qg, qo, f"quantize G={G}")
    # identical inputs: the moments agree exactly, only k's rounding matters
    st.update(P.compare_meta(Sg, kg, So, ko, f"quantize G={G}", state_rel=0.0))
    print(G, st)


def _dequant_tolerance(q, k):
    """Relative error bound of the fp32 un-expansion P * 2^(log2(|c|/448) / k).

    The exponent z = log2(|c|/448) / k is formed in fp32 (table value, 1/k and
    the product each round once: 3 half-ulps of |z|), 2^z comes from the SFU
    (2^-22 relative) and P and the final product round once each.
    """
    vals = oracle.e4m3_decode_all()
    mag = np.abs(vals[q])
    with np.errstate(divide="ignore"):
        z = np.where(mag > 0, np.abs(np.log2(np.where(mag > 0, mag, 1.0) / 448.0)), 0.0) / k
    return 2.0 ** -22 + 2.0 ** -23 + 3 * 2.0 ** -25 * z * math.log(2) * 2 + 2.0 ** -24


@pytest.mark.parametrize("G", [1, 16, 128, 256])
def test_dequantize_matches_oracle(G):
    x = _groups(G, max(64, 8192 // G), seed=100 + G)
    q, S, k = oracle.dre_quantize(x, G)
    xg = gpu_dequantize(q, S, k, G)
    xo = oracle.dre_dequantize(q, S, k, G)
    kk = np.repeat(k.astype(np.float64), G)[: q.size]
    tol = _dequant_tolerance(q, kk)
    rel = np.abs(xg.astype(np.float64) - xo) / np.where(xo != 0, np.abs(xo), 1.0)
    assert np.array_equal(xg == 0, xo == 0)
    assert np.array_equal(np.signbit(xg[xo != 0]), np.signbit(xo[xo != 0]))
    assert np.all(rel <= tol), f"worst rel {rel.max():.3e}"
    print(G, "dequant max rel", rel.max())


def test_all_256_codes_dequantize():
    codes = np.arange(256, dtype=np.uint8)
    codes = codes[(codes != 0x7F) & (codes != 0xFF)]
    for S, k in ((1.0 / 448, 1.0), (3e-12, 2.5), (7e-30, 5.0), (2e-3, 0.7)):
        Sa = np.array([S], np.float32)
        ka = np.array([k], np.float32)
        q = np.ascontiguousarray(codes)
        xg = gpu_dequantize(q, np.repeat(Sa, 1), np.repeat(ka, 1), 256)
        xo = oracle.dre_dequantize(q, Sa, ka, 256)
        tol = _dequant_tolerance(q, np.full(q.size, float(ka[0])))
        rel = np.abs(xg.astype(np.float64) - xo) / np.where(xo != 0, np.abs(xo), 1.0)
        assert np.all(rel <= tol), (S, k, rel.max())
        # the largest code dequantizes to (448 S)^(1/k)
        top = list(q).index(0x7E)
        assert abs(xg[top] / ((448.0 * float(Sa[0])) ** (1.0 / float(ka[0]))) - 1) < 3e-7


def test_round_trip_on_gpu():
    G = 128
    x = _groups(G, 256, seed=7)
    q, S, k = gpu_quantize(x, G)
    xr = gpu_dequantize(q, S, k, G)
    vals = oracle.e4m3_decode_all()
    for gi in range(256):
        sl = slice(G * gi, G * (gi + 1))
        xs = x[sl].astype(np.float64)
        mx = np.abs(xs).max()
        if mx == 0:
            assert not q[sl].any() and S[gi] == 0
            continue
        y = 448.0 * (np.abs(xs) / mx) ** float(k[gi])
        c = np.abs(vals[q[sl]])
        spacing = np.where(y < 2.0 ** -6, 2.0 ** -9, 2.0 ** (np.floor(np.log2(np.maximum(y, 1e-30))) - 3))
        assert np.all(np.abs(c - y) <= 0.5 * spacing * (1 + 1e-5) + 1e-9), gi
        nz = xs != 0
        assert np.all(np.sign(xr[sl][nz]) == np.sign(xs[nz]))
