"""The oracle's dequantized moments are correctly rounded to fp32, also where
the exact value lies right next to an fp32 rounding midpoint.

A dequantized moment is the fp32 value of sign(q) (|E4M3(q)| S)^(1/k) (COAT
review page, section 3: the dequantized tensor is X_FP32).  Where a group's
smallest |m_t| is the remainder of a partial cancellation, a one-ulp error in
that value becomes many ulps of m_t and moves k and S, so the parity of the
step rests on this rounding being right.  The reference here is a 50-digit
evaluation by mpmath, a library independent of the oracle.  The hard cases
lie within 1e-5 ulp (about 2^-41 relative) of a midpoint: closer than the
step kernel's double-float path resolves, far outside the oracle's own
float64 error.
"""
import numpy as np
import pytest

import oracle

mpmath = pytest.importorskip("mpmath")
mpmath.mp.dps = 50


def _correct_fp32(code, S, k, dec):
    mag = abs(dec[code])
    x = mpmath.power(mpmath.mpf(float(mag)) * mpmath.mpf(float(S)), 1 / mpmath.mpf(float(k)))
    f = np.float32(float(x))
    e = np.frexp(f)[1] - 24
    u = mpmath.ldexp(1, int(e))
    q = x / u
    n = mpmath.floor(q)
    r = q - n
    if r > 0.5 or (r == 0.5 and int(n) % 2 == 1):
        n += 1
    v = np.float32(float(n * u))
    return -v if code & 0x80 else v


def test_near_midpoint_values_round_correctly():
    dec = oracle.e4m3_decode_all()
    rng = np.random.default_rng(31)
    finite = np.array([c for c in range(1, 255) if c not in (0x7F, 0x80)], dtype=np.uint8)
    N = 4_000_000
    codes = rng.choice(finite, N)
    S = np.exp2(rng.uniform(-100.0, 0.0, N)).astype(np.float32)
    k = rng.uniform(0.6, 8.0, N).astype(np.float32)
    x = (np.abs(dec[codes]) * S.astype(np.float64)) ** (1.0 / k.astype(np.float64))
    ok = (x > 2.0 ** -126) & (x < 2.0 ** 127)
    ulp = np.spacing(x.astype(np.float32)).astype(np.float64)
    frac = x / ulp
    dist = np.abs(frac - np.floor(frac) - 0.5)
    hard = np.nonzero(ok & (dist < 1e-5))[0][:60]
    assert hard.size >= 20, "the search found too few values near a midpoint"
    easy = np.nonzero(ok)[0][:40]
    for idx in np.concatenate([hard, easy]):
        G = 1
        got = oracle.dre_dequantize(codes[idx:idx + 1], S[idx:idx + 1], k[idx:idx + 1], G)[0]
        want = _correct_fp32(int(codes[idx]), S[idx], k[idx], dec)
        assert got == want, (int(codes[idx]), float(S[idx]), float(k[idx]))


def _correct_k(mx, mn):
    """k = log R_E4M3 / log(max/min), below the cap, correctly rounded to fp32."""
    x = mpmath.log(mpmath.mpf(229376)) / mpmath.log(mpmath.mpf(float(mx)) / mpmath.mpf(float(mn)))
    f = np.float32(float(x))
    e = np.frexp(f)[1] - 24
    u = mpmath.ldexp(1, int(e))
    q = x / u
    n = mpmath.floor(q)
    r = q - n
    if r > 0.5 or (r == 0.5 and int(n) % 2 == 1):
        n += 1
    return np.float32(float(n * u))


def test_k_near_midpoints_rounds_correctly():
    rng = np.random.default_rng(32)
    N = 4_000_000
    mx = np.exp2(rng.uniform(-30.0, -2.0, N)).astype(np.float32)
    mn = (mx.astype(np.float64) * np.exp2(-rng.uniform(2.5, 40.0, N))).astype(np.float32)
    k = np.log(229376.0) / np.log(mx.astype(np.float64) / mn.astype(np.float64))
    ulp = np.spacing(k.astype(np.float32)).astype(np.float64)
    frac = k / ulp
    dist = np.abs(frac - np.floor(frac) - 0.5)
    # below the cap, and below the S-range guard's bound (S = max^k / 448 >= 2^-125)
    guard = (np.log2(448.0) - 125.0) / np.log2(mx.astype(np.float64))
    free = (k < 7.9) & (k < guard * (1 - 1e-6))
    hard = np.nonzero(free & (dist < 1e-5))[0][:40]
    assert hard.size >= 20, "the search found too few values of k near a midpoint"
    for idx in np.concatenate([hard, np.nonzero(free)[0][:20]]):
        group = np.array([mx[idx], mn[idx]], np.float32)
        got = oracle.dre_group(group)["k"]
        assert np.float32(got) == _correct_k(mx[idx], mn[idx]), (float(mx[idx]), float(mn[idx]))
