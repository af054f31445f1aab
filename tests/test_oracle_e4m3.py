"""Pins for the oracle's E4M3 codec (CPU only).

The codec is pinned against things other than itself: the OCP FP8 format's
named points (tests/golden/e4m3_ocp_points.txt), torch's float8_e4m3fn
conversion (a library routine, decoding and round-to-nearest-even encoding),
an independent argmin search, the midpoints between neighbouring codes and
saturation beyond 448.
"""
import math
import os

import numpy as np
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3_ocp_points.txt")


def _torch_decode_all():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_decode_matches_torch_float8_e4m3fn():
    ours = oracle.e4m3_decode_all()
    ref = _torch_decode_all()
    nan_ours = np.isnan(ours)
    assert np.array_equal(nan_ours, np.isnan(ref))
    assert list(np.nonzero(nan_ours)[0]) == [0x7F, 0xFF]
    assert np.array_equal(ours[~nan_ours], ref[~nan_ours])
    # sign of zero
    assert math.copysign(1.0, ours[0x80]) == -1.0


def test_decode_named_points_of_the_format():
    rows = 0
    with open(GOLDEN) as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            code, value, *_ = line.split()
            got = oracle.e4m3_decode(int(code, 16))
            if value == "nan":
                assert math.isnan(got), code
            else:
                assert got == float(value), (code, got, value)
                assert math.copysign(1.0, got) == math.copysign(1.0, float(value))
            rows += 1
    assert rows >= 10


def test_positive_codes_strictly_increasing_and_count():
    v = oracle.e4m3_decode_all()
    pos = v[1:127]
    assert len(pos) == 126 and np.all(pos > 0)
    assert np.all(np.diff(v[0:127]) > 0)
    assert v[0x7E] == 448.0 and v[0x01] == 2.0 ** -9
    # negative half mirrors the positive half
    assert np.array_equal(v[0x80:0xFF], -v[0x00:0x7F])


def test_encode_decode_identity_on_finite_codes():
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        d = oracle.e4m3_decode(c)
        want = 0x00 if c == 0x80 else c
        assert oracle.e4m3_encode(d) == want, hex(c)


def test_midpoints_round_to_even_mantissa():
    v = oracle.e4m3_decode_all()
    for c in range(0, 126):
        mid = 0.5 * (v[c] + v[c + 1])
        even = c if c % 2 == 0 else c + 1
        assert oracle.e4m3_encode(mid) == even, hex(c)
        assert oracle.e4m3_encode(-mid) == (0x80 | even if even else 0), hex(c)
        # just off the midpoint goes to the nearer neighbour
        eps = (v[c + 1] - v[c]) * 1e-6
        assert oracle.e4m3_encode(mid - eps) == c
        assert oracle.e4m3_encode(mid + eps) == c + 1


def test_saturation():
    for y in (448.0, 455.9, 464.0, 480.0, 1e6, 3.4e38):
        assert oracle.e4m3_encode(y) == 0x7E
        assert oracle.e4m3_encode(-y) == 0xFE
    assert oracle.e4m3_encode(1e-300) == 0
    assert oracle.e4m3_encode(-1e-300) == 0
    assert oracle.e4m3_encode(0.5 * 2.0 ** -9) == 0          # tie with zero -> even (zero)
    assert oracle.e4m3_encode(0.5 * 2.0 ** -9 * (1 + 1e-9)) == 1


def test_encode_equals_independent_argmin_brute_force():
    rng = np.random.default_rng(1234)
    n = 40000
    mag = np.exp2(rng.uniform(-12.0, 9.5, n))
    y = np.where(rng.random(n) < 0.5, -mag, mag).astype(np.float32).astype(np.float64)
    table = _torch_decode_all()[:127]  # finite non-negative values
    ours = oracle.e4m3_encode_array(y)
    d = np.abs(np.abs(y)[:, None] - table[None, :])
    best = d.min(axis=1, keepdims=True)
    cand = d == best
    # among equal distances pick the even code
    idx = np.where(cand & (np.arange(127)[None, :] % 2 == 0), np.arange(127)[None, :], 10**6).min(axis=1)
    idx = np.where(idx == 10**6, d.argmin(axis=1), idx)
    want = np.where((y < 0) & (idx != 0), 0x80 | idx, idx).astype(np.uint8)
    assert np.array_equal(ours, want)


def test_encode_matches_torch_rne_inside_range():
    rng = np.random.default_rng(99)
    n = 40000
    mag = np.exp2(rng.uniform(-11.0, np.log2(448.0), n))
    y = np.where(rng.random(n) < 0.5, -mag, mag).astype(np.float32)
    ours = oracle.e4m3_encode_array(y.astype(np.float64))
    ref = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ref = np.where(ref == 0x80, 0, ref)
    assert np.array_equal(ours, ref)
