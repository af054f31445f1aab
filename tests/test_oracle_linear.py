"""Pins of the oracle's FP8 linear layer with a per-group FP8 output
(oracle.linear_group_quantize).

COAT paper-review page, section 3: "mixed-granularity activation
quantization" (linear layers take per-tensor FP8 inputs) and "Triton
kernels", linear layer optimisation (the output tile is reshaped to
(BLOCK_M, BLOCK_N/G, G) and its maximum taken along the last axis).

The pins do not restate the oracle's formula: the product is checked against
exact rational arithmetic on E4M3 values decoded by torch, against a closed
form for rank-one inputs and against symmetries of the product; the output
quantization is checked against the separately pinned activation quantizer and
against invariances that fix the group axis.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

FINITE = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)


def torch_decode(codes: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def rn32(r: Fraction) -> float:
    """Round an exact rational to the nearest float32 (ties to even; normal range)."""
    if r == 0:
        return 0.0
    sign = -1 if r < 0 else 1
    a = abs(r)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    # 2^23 <= a / 2^(e-23) < 2^24
    while a >= Fraction(2) ** (e + 1):
        e += 1
    while a < Fraction(2) ** e:
        e -= 1
    scaled = a / Fraction(2) ** (e - 23)
    m = scaled.numerator // scaled.denominator
    rem = scaled - m
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and m % 2 == 1):
        m += 1
    return float(np.float32(sign * m * 2.0 ** (e - 23)))


def random_codes(rng, shape):
    return rng.choice(FINITE, size=shape)


@pytest.mark.parametrize("M,N,K", [(5, 8, 9), (9, 9, 9)])
def test_product_equals_exact_rationals(M, N, K):
    rng = np.random.default_rng(11 + M)
    G = 4 if N % 4 == 0 else 3 if N % 3 == 0 else 1
    xq, wq = random_codes(rng, (M, K)), random_codes(rng, (N, K))
    sx, sw = float(np.float32(0.0137)), float(np.float32(3.1e-3))
    y, _, _ = oracle.linear_group_quantize(xq, sx, wq, sw, G)
    X, W = torch_decode(xq), torch_decode(wq)
    for m in range(M):
        for n in range(N):
            s = sum(Fraction(float(X[m, k])) * Fraction(float(W[n, k])) for k in range(K))
            assert y[m, n] == rn32(Fraction(sx) * Fraction(sw) * s), (m, n)


def test_rank_one_closed_form():
    rng = np.random.default_rng(12)
    M, N, K, G = 6, 32, 96, 8
    c = random_codes(rng, M)
    d = random_codes(rng, N)
    xq = np.repeat(c[:, None], K, axis=1)
    wq = np.repeat(d[:, None], K, axis=1)
    sx, sw = float(np.float32(0.75)), float(np.float32(1.0 / 3.0))
    y, _, _ = oracle.linear_group_quantize(xq, sx, wq, sw, G)
    cv, dv = torch_decode(c), torch_decode(d)
    for m in range(M):
        for n in range(N):
            exact = Fraction(sx) * Fraction(sw) * K * Fraction(float(cv[m])) * Fraction(float(dv[n]))
            assert y[m, n] == rn32(exact)


def test_transpose_and_joint_permutation_of_k():
    rng = np.random.default_rng(13)
    M, N, K, G = 16, 48, 200, 16
    xq, wq = random_codes(rng, (M, K)), random_codes(rng, (N, K))
    y, _, _ = oracle.linear_group_quantize(xq, 0.5, wq, 0.25, G)
    yt, _, _ = oracle.linear_group_quantize(wq, 0.25, xq, 0.5, G)
    assert np.array_equal(y, yt.T)
    perm = rng.permutation(K)
    yp, _, _ = oracle.linear_group_quantize(xq[:, perm], 0.5, wq[:, perm], 0.25, G)
    assert np.array_equal(y, yp)


@pytest.mark.parametrize("G", [4, 16, 64])
def test_identity_weight_reduces_to_the_activation_quantizer(G):
    # W = I (code 0x38 = 1.0) and power-of-two scales: y = 2^a E4M3(xq) exactly,
    # a bf16 value, so the output must be the activation quantizer's on it
    rng = np.random.default_rng(14 + G)
    M, K = 12, 4 * G
    xq = random_codes(rng, (M, K))
    wq = np.zeros((K, K), np.uint8)
    np.fill_diagonal(wq, 0x38)
    sx, sw = 2.0 ** -3, 2.0 ** 5
    y, q, S = oracle.linear_group_quantize(xq, sx, wq, sw, G)
    expect = (torch_decode(xq) * 4.0).astype(np.float32)
    assert np.array_equal(y, expect)
    bits = (expect.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal((bits.astype(np.uint32) << 16).view(np.float32), expect)
    qa, _, Sa = oracle.act_quantize(bits, G)
    assert np.array_equal(q, qa) and np.array_equal(S, Sa)


def test_groups_run_along_rows():
    rng = np.random.default_rng(15)
    M, N, K, G = 16, 64, 40, 16
    xq, wq = random_codes(rng, (M, K)), random_codes(rng, (N, K))
    y, q, S = oracle.linear_group_quantize(xq, 0.01, wq, 0.02, G)
    assert S.shape == (M, N // G)
    # changing the weight rows of output group 2 changes only that group
    wq2 = wq.copy()
    wq2[2 * G:3 * G] = random_codes(rng, (G, K))
    y2, q2, S2 = oracle.linear_group_quantize(xq, 0.01, wq2, 0.02, G)
    keep = np.ones(N, bool)
    keep[2 * G:3 * G] = False
    assert np.array_equal(q[:, keep], q2[:, keep])
    assert np.array_equal(np.delete(S, 2, axis=1), np.delete(S2, 2, axis=1))
    assert not np.array_equal(S[:, 2], S2[:, 2])
    # changing one input row changes only that row's groups
    xq2 = xq.copy()
    xq2[5] = random_codes(rng, K)
    _, q3, S3 = oracle.linear_group_quantize(xq2, 0.01, wq, 0.02, G)
    assert np.array_equal(np.delete(q, 5, axis=0), np.delete(q3, 5, axis=0))
    assert np.array_equal(np.delete(S, 5, axis=0), np.delete(S3, 5, axis=0))


def test_power_of_two_input_scale_moves_only_the_output_scales():
    rng = np.random.default_rng(16)
    M, N, K, G = 8, 32, 24, 8
    xq, wq = random_codes(rng, (M, K)), random_codes(rng, (N, K))
    y, q, S = oracle.linear_group_quantize(xq, 0.3, wq, 0.07, G)
    y2, q2, S2 = oracle.linear_group_quantize(xq, 0.3 * 8, wq, 0.07, G)
    assert np.array_equal(y2, y * 8) and np.array_equal(S2, S * 8) and np.array_equal(q2, q)


def test_rejects_bad_shapes():
    with pytest.raises(ValueError):
        oracle.linear_group_quantize(np.zeros((4, 8), np.uint8), 1.0, np.zeros((16, 9), np.uint8), 1.0, 4)
    with pytest.raises(ValueError):
        oracle.linear_group_quantize(np.zeros((4, 8), np.uint8), 1.0, np.zeros((12, 8), np.uint8), 1.0, 8)


# ---------------------------------------------------------------------------
# the pins above reject plausible mistakes (planted in scratch variants)
# ---------------------------------------------------------------------------

def _variant(kind):
    def f(xq, sx, wq, sw, G, nthreads=0):
        xq = np.ascontiguousarray(xq, dtype=np.uint8)
        wq = np.ascontiguousarray(wq, dtype=np.uint8)
        M, K = xq.shape
        N, K2 = wq.shape
        if K != K2 or N % G:
            raise ValueError("bad shapes")
        dec = oracle.e4m3_decode_all()
        acc = dec[xq] @ dec[wq].T
        scale = np.float64(np.float32(sx)) * np.float64(np.float32(sw))
        if kind == "no_sw":
            scale = np.float64(np.float32(sx))
        elif kind == "sx_over_sw":
            scale = np.float64(np.float32(sx)) / np.float64(np.float32(sw))
        elif kind == "acc_rounded_first":
            acc = acc.astype(np.float32).astype(np.float64)
        elif kind == "w_not_transposed":
            if K != N:
                raise NotImplementedError
            acc = dec[xq] @ dec[wq]
        elif kind == "output_transposed":
            if M != N:
                raise NotImplementedError
            acc = acc.T
        y = (scale * acc).astype(np.float32)
        if kind == "groups_down_columns":
            if M % G:
                raise NotImplementedError
            qt, St = oracle.absmax_quantize(np.ascontiguousarray(y.T), G, nthreads)
            return y, qt.reshape(N, M).T.copy(), St.reshape(N, M // G).T.copy()
        q, S = oracle.absmax_quantize(y, G, nthreads)
        return y, q.reshape(M, N), S.reshape(M, N // G)
    return f


PINS = [lambda: test_product_equals_exact_rationals(5, 8, 9),
        lambda: test_product_equals_exact_rationals(9, 9, 9), test_rank_one_closed_form,
        test_transpose_and_joint_permutation_of_k,
        lambda: test_identity_weight_reduces_to_the_activation_quantizer(16),
        test_groups_run_along_rows, test_power_of_two_input_scale_moves_only_the_output_scales]


@pytest.mark.parametrize("kind", ["no_sw", "sx_over_sw", "acc_rounded_first", "groups_down_columns",
                                  "w_not_transposed", "output_transposed"])
def test_pins_reject_planted_mistakes(kind, monkeypatch):
    monkeypatch.setattr(oracle, "linear_group_quantize", _variant(kind))
    caught = 0
    for pin in PINS:
        try:
            pin()
        except NotImplementedError:
            pass                      # the mistake needs another shape
        except Exception:
            caught += 1
    assert caught >= 1, f"no pin rejects the '{kind}' variant"


def test_unplanted_variant_passes_every_pin(monkeypatch):
    monkeypatch.setattr(oracle, "linear_group_quantize", _variant("none"))
    for pin in PINS:
        pin()
