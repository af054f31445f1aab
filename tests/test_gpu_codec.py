"""GPU parity of the standalone DRE quantizer / dequantizer against the oracle."""

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


@pytest.mark.parametrize("G", [32, 128, 256])
def test_quantize_several_tiles_per_cta(G):
    """A buffer of more than three tiles of 4096 elements for each of eight
    CTAs per SM, with a ragged last tile and a few all-zero and one-non-zero
    groups: the quantizer's persistent form (G >= 32) takes several tiles per
    CTA; codes, S and k against the oracle over the whole buffer."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    n = 3 * 8 * sms * 4096 + 5 * G + G // 2 + 7
    ng = (n + G - 1) // G
    rng = np.random.default_rng(300 + G)
    s = 10.0 ** rng.uniform(-12, 2, ng)
    x = (rng.standard_normal(ng * G) * np.repeat(s, G))[:n].astype(np.float32)
    x[:4 * G] = 0.0
    x[4 * G + 3] = 1.5
    x[5 * G:6 * G] = 0.0
    x[6 * G] = -2.0e-30
    qg, Sg, kg = gpu_quantize(x, G)
    qo, So, ko = oracle.dre_quantize(x, G)
    st = P.compare_codes(qg, qo, f"many tiles G={G}")
    st.update(P.compare_meta(Sg, kg, So, ko, f"many tiles G={G}", state_rel=0.0))
    print(G, st)


# The dequantizer's bar: within 1e-6 relative of the oracle's correctly
# rounded fp32 value (the bar of the step's weights, scales and exponents),
# or one fp32 subnormal step for results below 2^-126, which are scaled with a
# second rounding.
DEQUANT_RTOL = 1e-6
SUBNORMAL_STEP = 2.0 ** -149


def _dequant_ok(xg, xo):
    err = np.abs(xg.astype(np.float64) - xo.astype(np.float64))
    return (err <= DEQUANT_RTOL * np.abs(xo.astype(np.float64))) | (
        (np.abs(xo) < 2.0 ** -126) & (err <= SUBNORMAL_STEP))


@pytest.mark.parametrize("G", [1, 2, 4, 8, 16, 128, 256])
def test_dequantize_matches_oracle(G):
    x = _groups(G, max(64, 8192 // G), seed=100 + G)
    q, S, k = oracle.dre_quantize(x, G)
    xg = gpu_dequantize(q, S, k, G)
    xo = oracle.dre_dequantize(q, S, k, G)
    rel = np.abs(xg.astype(np.float64) - xo) / np.where(xo != 0, np.abs(xo), 1.0)
    assert np.array_equal(xg == 0, xo == 0)
    assert np.array_equal(np.signbit(xg[xo != 0]), np.signbit(xo[xo != 0]))
    ok = _dequant_ok(xg, xo)
    assert ok.all(), f"{int((~ok).sum())} values off; worst rel {rel.max():.3e}"
    print(G, "dequant max rel", rel.max(), "bit-equal", float((xg == xo).mean()))


def test_all_256_codes_dequantize():
    codes = np.arange(256, dtype=np.uint8)
    codes = codes[(codes != 0x7F) & (codes != 0xFF)]
    for S, k in ((1.0 / 448, 1.0), (3e-12, 2.5), (7e-30, 5.0), (2e-3, 0.7)):
        Sa = np.array([S], np.float32)
        ka = np.array([k], np.float32)
        q = np.ascontiguousarray(codes)
        xg = gpu_dequantize(q, np.repeat(Sa, 1), np.repeat(ka, 1), 256)
        xo = oracle.dre_dequantize(q, Sa, ka, 256)
        rel = np.abs(xg.astype(np.float64) - xo) / np.where(xo != 0, np.abs(xo), 1.0)
        assert _dequant_ok(xg, xo).all(), (S, k, rel.max())
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


def test_dequantize_extreme_scales_and_exponents():
    """Every code under (S, k) pairs spread over the whole stored range,
    including compressions (k < 1) and results that leave the normal range."""
    codes = np.arange(256, dtype=np.uint8)
    codes = np.ascontiguousarray(codes[(codes != 0x7F) & (codes != 0xFF)])
    rng = np.random.default_rng(5)
    pairs = [(2.0 ** -125, 1.0), (2.0 ** 126, 8.0), (2.0 ** -125, 8.0), (3e-30, 0.6),
             (1e20, 0.9)] + [(float(2.0 ** rng.uniform(-125, 60)), float(rng.uniform(0.6, 8.0)))
                             for _ in range(40)]
    for S, k in pairs:
        Sa = np.array([S], np.float32)
        ka = np.array([k], np.float32)
        xo = oracle.dre_dequantize(codes, Sa, ka, 256)
        if not np.all(np.isfinite(xo)):
            continue
        xg = gpu_dequantize(codes, Sa, ka, 256)
        ok = _dequant_ok(xg, xo)
        assert ok.all(), (S, k, int((~ok).sum()))


def _hard_k_pairs(count, seed):
    """(max, min) pairs whose exact k lies within 1e-5 ulp of an fp32
    rounding midpoint (found by search in float64), below the cap."""
    rng = np.random.default_rng(seed)
    N = 3_000_000
    mx = np.exp2(rng.uniform(-40.0, 10.0, N)).astype(np.float32)
    mn = (mx.astype(np.float64) * np.exp2(-rng.uniform(2.3, 40.0, N))).astype(np.float32)
    kk = np.log(229376.0) / np.log(mx.astype(np.float64) / mn.astype(np.float64))
    frac = kk / np.spacing(kk.astype(np.float32)).astype(np.float64)
    dist = np.abs(frac - np.floor(frac) - 0.5)
    hard = np.nonzero((kk < 7.9) & (dist < 1e-5))[0][:count]
    return mx[hard], mn[hard]


@pytest.mark.parametrize("G", [2, 128])
def test_quantize_k_at_hard_roundings(G):
    """Groups whose k lies within 1e-5 ulp of an fp32 midpoint: the codec's k
    is the oracle's correctly rounded value, bit for bit."""
    mx, mn = _hard_k_pairs(64, seed=50 + G)
    assert mx.size >= 30
    rng = np.random.default_rng(G)
    groups = []
    for a, b in zip(mx, mn):
        x = np.exp(rng.uniform(np.log(float(b)), np.log(float(a)), G)).astype(np.float32)
        x[0], x[-1] = a, b
        groups.append(x * np.where(rng.random(G) < 0.5, -1, 1).astype(np.float32))
    x = np.concatenate(groups).astype(np.float32)
    qg, Sg, kg = gpu_quantize(x, G)
    qo, So, ko = oracle.dre_quantize(x, G)
    assert np.array_equal(kg.view(np.uint32), ko.view(np.uint32))
    P.compare_meta(Sg, kg, So, ko, f"hard k G={G}", state_rel=0.0)
    P.compare_codes(qg, qo, f"hard k G={G}")

