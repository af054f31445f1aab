"""The comparison helpers of the GPU parity tests accept what the tolerances
allow and reject what they do not.  The deviations are planted, on the CPU,
into a real oracle step's output."""
import numpy as np
import pytest

import oracle
from coat_fp8_adamw_gb300 import synth

import _parity as P


@pytest.fixture(scope="module")
def step_output():
    G, n = 128, 128 * 512
    mq, vq, meta = P.adamw_like_state(n, G, seed=5, oracle=oracle)
    rng = np.random.default_rng(6)
    w = (rng.standard_normal(n) * 0.02).astype(np.float32)
    g = synth.f32_to_bf16_bits((rng.standard_normal(n) * 1e-3).astype(np.float32))
    hp = synth.HYPER
    oracle.adamw_step(w, g, mq, vq, meta, G, hp["beta1"], hp["beta2"], hp["lr"], hp["eps"],
                      hp["weight_decay"], 3)
    return w, mq, vq, meta


def test_identical_outputs_pass(step_output):
    w, mq, vq, meta = step_output
    P.compare_w(w.copy(), w)
    assert P.compare_codes(mq.copy(), mq, "m")["flips"] == 0
    r = P.compare_meta(meta[:, 0].copy(), meta[:, 1].copy(), meta[:, 0], meta[:, 1], "m")
    assert r["k_bit_equal_frac"] == 1.0 and r["S_bit_equal_frac"] == 1.0


def _step_code(c: int, up: bool) -> int:
    """The adjacent code one grid step further from (up) or closer to zero."""
    o = int(P.code_ordinal(np.array([c]))[0]) + (1 if up else -1) * (1 if c < 128 else -1)
    return o if o >= 0 else 128 | -o


def test_codes_one_step_apart_in_few_places_pass(step_output):
    _, mq, _, _ = step_output
    bad = mq.copy()
    idx = np.nonzero((mq & 0x7F) > 1)[0][:5]          # 5 of 65536 < 1e-4
    for i in idx:
        bad[i] = _step_code(int(mq[i]), up=False)
    assert P.compare_codes(bad, mq, "m")["flips"] == 5


def test_code_two_steps_apart_fails(step_output):
    _, mq, _, _ = step_output
    bad = mq.copy()
    i = int(np.nonzero((mq & 0x7F) > 2)[0][0])
    bad[i] = _step_code(_step_code(int(mq[i]), up=False), up=False)
    with pytest.raises(AssertionError, match="differs by 2"):
        P.compare_codes(bad, mq, "m")


def test_sign_flip_fails(step_output):
    _, mq, _, _ = step_output
    bad = mq.copy()
    small = np.nonzero((mq & 0x7F) != 0)[0]
    i = int(small[np.argmin(mq[small] & 0x7F)])       # the smallest non-zero magnitude
    bad[i] = mq[i] ^ 0x80
    with pytest.raises(AssertionError):
        P.compare_codes(bad, mq, "m")


def test_too_many_one_step_flips_fail(step_output):
    _, mq, _, _ = step_output
    bad = mq.copy()
    idx = np.nonzero((mq & 0x7F) > 1)[0][:20]          # 20 of 65536 > 1e-4
    for i in idx:
        bad[i] = _step_code(int(mq[i]), up=False)
    with pytest.raises(AssertionError, match="of codes differ"):
        P.compare_codes(bad, mq, "m")


def test_weight_tolerance(step_output):
    w = step_output[0]
    i = int(np.argmax(np.abs(w)))
    ok = w.copy()
    ok[i] = np.float32(w[i] * (1 + 5e-7))
    P.compare_w(ok, w)
    bad = w.copy()
    bad[i] = np.float32(w[i] * (1 + 2e-6))
    with pytest.raises(AssertionError, match="outside tolerance"):
        P.compare_w(bad, w)
    # the absolute floor admits 1e-9 near zero, not more
    z = np.zeros(4, np.float32)
    P.compare_w(np.full(4, 5e-10, np.float32), z)
    with pytest.raises(AssertionError):
        P.compare_w(np.full(4, 2e-9, np.float32), z)


@pytest.mark.parametrize("col", [0, 1])
def test_scale_and_exponent_tolerance(step_output, col):
    meta = step_output[3]
    S, k = meta[:, 0].copy(), meta[:, 1].copy()
    j = int(np.nonzero(S > 0)[0][0])
    x = (S if col == 0 else k)
    x[j] = np.float32(x[j] * (1 + 2e-6))
    with pytest.raises(AssertionError):
        P.compare_meta(S, k, meta[:, 0], meta[:, 1], "m")
    x[j] = (meta[:, col])[j] * np.float32(1 + 4e-7)
    P.compare_meta(S, k, meta[:, 0], meta[:, 1], "m")


def test_zero_scale_mismatch_fails(step_output):
    meta = step_output[3]
    S = meta[:, 0].copy()
    S[int(np.nonzero(S > 0)[0][0])] = 0.0
    with pytest.raises(AssertionError, match="zero scales differ"):
        P.compare_meta(S, meta[:, 1], meta[:, 0], meta[:, 1], "m")
