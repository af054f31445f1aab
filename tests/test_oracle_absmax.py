"""Pins of the oracle's FP8 quantization without the expansion (the no-DRE arm
of the quantization-error comparison): S = max|X| / 448, q = E4M3(X / S)
(COAT review page, section 3, FP8 quantization equation).

The pins do not re-type the oracle's formula: exact recovery of values built
on the E4M3 grid, torch's own E4M3 conversion, the round-trip error bound of
the format, and the special groups.
"""
import numpy as np
import pytest
import torch

import oracle


def _decode_all():
    return np.array([oracle.e4m3_decode(c) for c in range(256)])


def test_groups_on_the_grid_are_recovered_exactly():
    rng = np.random.default_rng(1)
    dec = _decode_all()
    G = 64
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)])
    codes = rng.choice(finite, size=(40, G))
    codes[:, 0] = 0x7E                              # every group reaches 448
    scale = 2.0 ** rng.integers(-30, 10, size=40)   # power of two: max / 448 is exact
    x = (dec[codes] * scale[:, None]).astype(np.float32).ravel()
    q, S = oracle.absmax_quantize(x, G)
    assert np.array_equal(S, scale.astype(np.float32))
    expect = codes.ravel().astype(np.uint8)
    expect[expect == 0x80] = 0x00                   # -0 encodes as +0
    assert np.array_equal(q, expect)


def test_agrees_with_torch_e4m3_conversion():
    rng = np.random.default_rng(2)
    G = 128
    x = (rng.standard_normal(128 * 200) * 10.0 ** rng.uniform(-8, 3, 128 * 200)).astype(np.float32)
    q, S = oracle.absmax_quantize(x, G)
    y = x.reshape(-1, G).astype(np.float64) / S.astype(np.float64)[:, None]
    assert np.all(np.abs(y) <= 448.0 * (1 + 2.0 ** -23))
    y32 = np.clip(y.astype(np.float32), -448.0, 448.0)
    tq = torch.from_numpy(y32.ravel()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    tq = np.where(tq == 0x80, 0, tq)
    diff = np.nonzero(tq != q)[0]
    # torch rounds the float32 quotient, the oracle the exact one: they may only
    # differ where the float32 rounding landed exactly on a midpoint of the grid
    dec = _decode_all()
    for i in diff:
        a, b = dec[q[i]], dec[tq[i]]
        assert abs(float(y32.ravel()[i]) - (a + b) / 2) == 0.0
    assert diff.size <= 2


def test_round_trip_error_within_half_a_grid_step():
    rng = np.random.default_rng(3)
    G = 32
    x = (rng.standard_normal(32 * 500) * 10.0 ** rng.uniform(-5, 0, 32 * 500)).astype(np.float32)
    q, S = oracle.absmax_quantize(x, G)
    dec = _decode_all()
    y = np.abs(x.reshape(-1, G).astype(np.float64) / S.astype(np.float64)[:, None]).ravel()
    back = np.abs(dec[q]).astype(np.float64)
    # E4M3: 3 mantissa bits, exponent 2^-6 .. 2^8, subnormal spacing 2^-9
    e = np.floor(np.log2(np.maximum(y, 2.0 ** -6)))
    half_step = np.where(y < 2.0 ** -6, 2.0 ** -10, 2.0 ** (e - 4))
    assert np.all(np.abs(back - y) <= half_step * (1 + 1e-9))


def test_special_groups():
    G = 16
    zero = np.zeros(G, np.float32)
    one = np.zeros(G, np.float32)
    one[3] = -2.5e-3
    x = np.concatenate([zero, one, np.full(5, 7.0, np.float32)])   # ragged last group
    q, S = oracle.absmax_quantize(x, G)
    assert S[0] == 0 and not q[:G].any()
    assert S[1] == np.float32(2.5e-3 / 448) and q[G + 3] == 0xFE and np.count_nonzero(q[G:2 * G]) == 1
    assert S[2] == np.float32(7.0 / 448) and np.all(q[2 * G:] == 0x7E)


def test_bad_arguments():
    with pytest.raises(ValueError):
        oracle.absmax_quantize(np.zeros(0, np.float32), 16)


def test_activation_groups_run_along_rows():
    """The activation quantizer groups G consecutive columns of one row; its
    second output is the first one transposed."""
    rng = np.random.default_rng(4)
    M, N, G = 32, 64, 16
    row_scale = 2.0 ** rng.integers(-20, 5, size=(M, N // G))     # one magnitude per row group
    x = np.repeat(row_scale, G, axis=1) * rng.uniform(-1, 1, size=(M, N))
    x[:, ::G] = np.repeat(row_scale, 1, axis=1) * 448 / 256       # a known max in each group
    bits = (x.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)   # truncate to bf16
    xb = (bits.astype(np.uint32) << 16).view(np.float32)
    q, qt, S = oracle.act_quantize(bits, G)
    expect_S = (np.abs(xb).reshape(M, N // G, G).max(axis=2).astype(np.float64) / 448).astype(np.float32)
    assert np.array_equal(S, expect_S)
    assert np.array_equal(qt, q.T)
    # each group's largest element sits at the top of the grid
    assert np.all(np.abs(q.reshape(M, N // G, G).astype(int) & 0x7F).max(axis=2) == 0x7E)
