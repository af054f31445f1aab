"""The activation quantizer forms each group's scale RN(max / 448) without a
division: q = RN(max y) with y = RN(1/448), then one FMA correction from the
exact remainder max - 448 q (Markstein's division by a known divisor).  The
group maximum of a bf16 activation is itself a bf16 value, so the method is
checked here, in exact rational arithmetic with one rounding per operation,
against the correctly rounded quotient for every non-negative finite bf16
value, subnormals included."""
from fractions import Fraction

import numpy as np


def _rn32(a: Fraction) -> Fraction:
    """Nearest float32 to a non-negative rational (ties to even), subnormals included."""
    if a == 0:
        return Fraction(0)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    ulp = Fraction(2) ** (max(e, -126) - 23)
    q, rem = divmod(a, ulp)
    if 2 * rem > ulp or (2 * rem == ulp and q % 2 == 1):
        q += 1
    return q * ulp


def test_rounding_helper_matches_numpy_float32():
    rng = np.random.default_rng(0)
    for v in rng.random(200) * 10.0 ** rng.integers(-40, 38, 200):
        assert _rn32(Fraction(float(v))) == Fraction(float(np.float32(v)))


def test_fma_corrected_quotient_is_correctly_rounded_for_every_bf16():
    y = _rn32(Fraction(1, 448))
    assert y == Fraction(float(np.float32(1.0) / np.float32(448.0)))
    bits = np.arange(0, 0x7F80, dtype=np.uint32) << 16          # every finite bf16 >= 0
    for x in bits.view(np.float32):
        m = Fraction(float(x))
        q = _rn32(m * y)
        r = m - 448 * q                                          # exact in one FMA: |r| is tiny
        r = _rn32(r) if r >= 0 else -_rn32(-r)
        s = r * y + q
        got = _rn32(s) if s >= 0 else -_rn32(-s)
        assert got == _rn32(m / 448), float(m)
