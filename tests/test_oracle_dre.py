"""Pins for the oracle's Dynamic Range Expansion quantizer (CPU only).

Pinned against: hand-derived worked examples (tests/golden), the identity
R_X^k = R_E4M3 of the optimal exponent (COAT paper-review page, section 3,
Dynamic Range Expansion), k found by bisection on that identity without
logarithms, the k = 1 special case which is plain absmax quantization (the
FP8 quantization equation) as done by torch's float8_e4m3fn conversion,
invariances (sign, permutation, exact power-of-two scaling), the round-trip
error bound of the E4M3 grid, and ragged tails.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle

R = oracle.R_E4M3_DEFAULT
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "dre_worked_examples.txt")


def _parse_value(tok: str) -> float:
    if "*" in tok:
        a, b = tok.split("*")
        return _parse_value(a) * _parse_value(b)
    if tok.startswith("-"):
        return -_parse_value(tok[1:])
    if tok.startswith("2^"):
        return 2.0 ** int(tok[2:])
    return float(tok)


def _parse_expr(tok: str) -> float:
    safe = {"log2": math.log2}
    return float(eval(tok.replace("^", "**"), {"__builtins__": {}}, safe))


def _golden_examples():
    blocks, cur = [], {}
    with open(GOLDEN) as fh:
        for raw in fh:
            line = raw.split("#", 1)[0].strip()
            if not line:
                continue
            key, rest = line.split(None, 1)
            if key == "name" and cur:
                blocks.append(cur)
                cur = {}
            cur[key] = rest.strip()
    if cur:
        blocks.append(cur)
    return blocks


EXAMPLES = _golden_examples()


@pytest.mark.parametrize("ex", EXAMPLES, ids=[e["name"] for e in EXAMPLES])
def test_worked_examples(ex):
    x = np.array([_parse_value(t) for t in ex["x"].split()], dtype=np.float32)
    r = oracle.dre_group(x, float(ex["R"]))
    want_q = [int(t, 16) for t in ex["q"].split()]
    assert list(r["q"]) == want_q
    k_want = _parse_expr(ex["k"])
    assert r["k"] == np.float32(k_want)
    S_want = _parse_expr(ex["S"])
    if S_want == 0:
        assert r["S"] == 0
    else:
        assert abs(float(r["S"]) - S_want) <= 2e-5 * S_want


def _random_groups(count, G, seed):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(count):
        scale = 10.0 ** rng.uniform(-9, 1)
        kind = rng.integers(0, 3)
        if kind == 0:
            x = rng.standard_normal(G) * scale
        elif kind == 1:
            x = rng.standard_normal(G) ** 2 * scale
        else:
            x = np.exp(rng.uniform(-4, 0, G)) * scale * np.sign(rng.standard_normal(G))
        out.append(x.astype(np.float32))
    return out


def test_expanded_range_equals_R_E4M3_when_uncapped():
    n_uncapped = 0
    for x in _random_groups(300, 128, 5):
        r = oracle.dre_group(x, R)
        a = np.abs(x.astype(np.float64))
        mx, mn = a.max(), a[a > 0].min()
        if r["k_exact"] != r["k_formula"]:
            continue  # cap or guard active
        n_uncapped += 1
        # R_X^k = R_E4M3 at the exact k
        assert abs(math.pow(mx / mn, r["k_exact"]) / R - 1.0) < 1e-12
        # with the stored fp32 k the expanded range is within the rounding of k
        y = np.abs(r["y"])
        ratio = y.max() / y[y > 0].min()
        assert abs(ratio / R - 1.0) < math.log(R) * 2.0 ** -23
        # the group max lands on 448, the group min on the smallest subnormal
        assert r["q"][np.argmax(a)] & 0x7F == 0x7E
        assert r["q"][np.argmin(np.where(a > 0, a, np.inf))] & 0x7F == 0x01
    assert n_uncapped > 200


def test_min_lands_on_min_normal_with_the_other_reading_of_R():
    for x in _random_groups(50, 64, 6):
        r = oracle.dre_group(x, oracle.R_E4M3_MIN_NORMAL)
        if r["k_exact"] != r["k_formula"]:
            continue
        a = np.abs(x)
        assert r["q"][np.argmin(np.where(a > 0, a, np.inf))] & 0x7F == 0x08


def _bisect_k(rx: float, target: float) -> float:
    lo, hi = 1e-3, 1e2
    for _ in range(400):
        mid = 0.5 * (lo + hi)
        if math.pow(rx, mid) < target:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


def test_k_formula_equals_bisection():
    for x in _random_groups(60, 32, 7):
        r = oracle.dre_group(x, R)
        a = np.abs(x.astype(np.float64))
        rx = a.max() / a[a > 0].min()
        kb = _bisect_k(rx, R)
        assert abs(r["k_formula"] / kb - 1.0) < 1e-11


def test_cap_and_guard():
    for x in _random_groups(200, 16, 8):
        r = oracle.dre_group(x, R)
        assert 0 < r["k"] <= 8.0
        assert r["k_exact"] <= r["k_formula"] + 1e-15
        S = float(r["S"])
        assert 2.0 ** -125 * (1 - 1e-5) <= S <= 2.0 ** 126
        # S = max^k / 448 at the stored k
        mx = float(np.abs(x).max())
        assert abs(S / (mx ** float(r["k"]) / 448.0) - 1.0) < 2.0 ** -23


def test_k_one_is_plain_absmax_quantization():
    """With R_X = R the optimal k is 1 and DRE reduces to the FP8 quantization equation."""
    R2 = 2.0 ** 18
    rng = np.random.default_rng(11)
    for _ in range(50):
        x = rng.standard_normal(64).astype(np.float32)
        x[0], x[1] = 1.0, 2.0 ** -18  # fixes max 1 and min 2^-18 -> R_X = R2
        x = np.where(np.abs(x) > 1.0, np.sign(x) * 0.999, x).astype(np.float32)
        x = np.where((np.abs(x) < 2.0 ** -18) & (x != 0), 2.0 ** -17, x).astype(np.float32)
        x[0], x[1] = 1.0, 2.0 ** -18
        r = oracle.dre_group(x, R2)
        assert r["k"] == 1.0
        S = np.float64(np.float32(1.0 / 448.0))
        assert float(r["S"]) == S
        ref = torch.from_numpy(x.astype(np.float64) * 448.0).to(torch.float8_e4m3fn)
        ref = ref.view(torch.uint8).numpy()
        ref = np.where(ref == 0x80, 0, ref)
        assert np.array_equal(r["q"], ref)


def test_sign_and_permutation_symmetry():
    rng = np.random.default_rng(12)
    for x in _random_groups(40, 128, 9):
        r = oracle.dre_group(x, R)
        rn = oracle.dre_group(-x, R)
        assert rn["k"] == r["k"] and rn["S"] == r["S"]
        nz = r["q"] != 0
        assert np.array_equal(rn["q"][nz], r["q"][nz] ^ 0x80)
        perm = rng.permutation(x.size)
        rp = oracle.dre_group(x[perm], R)
        assert rp["k"] == r["k"] and rp["S"] == r["S"]
        assert np.array_equal(rp["q"], r["q"][perm])


def test_power_of_two_scaling_invariance():
    for x in _random_groups(40, 64, 10):
        a = np.abs(x)
        if a.max() > 2.0 ** 20 or a[a > 0].min() < 2.0 ** -100:
            continue
        r = oracle.dre_group(x, R)
        if r["k_exact"] != r["k_formula"]:
            continue
        xs = (x * np.float32(2.0 ** -3)).astype(np.float32)
        rs = oracle.dre_group(xs, R)
        if rs["k_exact"] != rs["k_formula"]:
            continue
        assert rs["k"] == r["k"]
        assert np.array_equal(rs["q"], r["q"])
        want = float(r["S"]) * 2.0 ** (-3.0 * float(r["k"]))
        assert abs(float(rs["S"]) / want - 1.0) < 2.0 ** -22


def test_dequantize_round_trip_within_grid_error():
    x = np.concatenate(_random_groups(64, 128, 13))
    q, S, k = oracle.dre_quantize(x, 128)
    xd = oracle.dre_dequantize(q, S, k, 128)
    vals = oracle.e4m3_decode_all()
    for g in range(64):
        sl = slice(128 * g, 128 * (g + 1))
        xg, dg = x[sl].astype(np.float64), xd[sl].astype(np.float64)
        mx = np.abs(xg).max()
        kk = float(k[g])
        y = 448.0 * (np.abs(xg) / mx) ** kk
        code_val = np.abs(vals[q[sl]])
        # the code is the grid point nearest to y: within half the local spacing
        spacing = np.where(y < 2.0 ** -6, 2.0 ** -9, 2.0 ** (np.floor(np.log2(np.maximum(y, 1e-30))) - 3))
        assert np.all(np.abs(code_val - y) <= 0.5 * spacing * (1 + 1e-9) + 1e-12)
        # dequantization inverts the expansion: x_hat = (code * S)^(1/k) = mx (code/448)^(1/k)
        want = mx * (code_val / 448.0) ** (1.0 / kk)
        assert np.allclose(np.abs(dg), want, rtol=2e-6, atol=0)
        assert np.all(np.sign(dg[xg != 0]) == np.sign(xg[xg != 0]))


def test_ragged_tail_group_is_quantized_on_its_own():
    rng = np.random.default_rng(14)
    x = (rng.standard_normal(1000) * 1e-3).astype(np.float32)
    q, S, k = oracle.dre_quantize(x, 128)
    assert S.size == 8
    tail = oracle.dre_group(x[896:], R)
    assert np.array_equal(q[896:], tail["q"])
    assert S[7] == tail["S"] and k[7] == tail["k"]
    head = oracle.dre_group(x[:128], R)
    assert np.array_equal(q[:128], head["q"])
