"""Comparison helpers for the GPU-vs-oracle parity tests.

Tolerances (floating point, from the stated targets of this port):
  * master weights: |w_gpu - w_ref| <= 1e-6 |w_ref| + 1e-9;
  * E4M3 codes: at most 1e-4 of the codes differ, each by one step of the
    E4M3 grid (adjacent codes of the same sign, or 0x00 / +-0x01);
  * k: relative 1e-6;
  * S: relative 1e-6.  S = max^k / 448 is ill-conditioned in the group's
    extreme moments (condition number up to ~30), so this holds only because
    the kernel re-evaluates those extremes exactly; ``s_condition`` gives the
    sensitivity for diagnostics.
"""
from __future__ import annotations

import numpy as np

W_RTOL = 1e-6
W_ATOL = 1e-9
CODE_FLIP_FRAC = 1e-4
K_RTOL = 1e-6
S_RTOL = 1e-6
# agreement of the fp32 moments between an fp32 GPU evaluation and the float64
# oracle rounded to fp32: a few units in the last place
STATE_REL = 4 * 2.0 ** -24
# stored k agreement
K_REL = 2 * 2.0 ** -24
R_E4M3 = 448.0 * 512.0


def code_ordinal(c: np.ndarray) -> np.ndarray:
    c = c.astype(np.int64)
    return np.where(c >= 128, -(c & 127), c)


def compare_codes(gpu: np.ndarray, ref: np.ndarray, what: str) -> dict:
    """Codes within one E4M3 step of the oracle's, few of them off; a zero is
    always stored as 0x00, never 0x80."""
    assert not (gpu == 0x80).any(), f"{what}: a zero stored as 0x80"
    d = np.abs(code_ordinal(gpu) - code_ordinal(ref))
    frac = float((d > 0).mean()) if d.size else 0.0
    assert d.size == 0 or d.max() <= 1, f"{what}: a code differs by {d.max()} E4M3 steps"
    assert frac <= CODE_FLIP_FRAC, f"{what}: {frac:.3e} of codes differ (> {CODE_FLIP_FRAC})"
    return {"flip_frac": frac, "flips": int((d > 0).sum())}


def assert_codes_equal(gpu: np.ndarray, ref: np.ndarray, what: str) -> None:
    """Bit-identical codes (the quantizers whose input is the oracle's own)."""
    bad = np.nonzero(gpu.ravel() != ref.ravel())[0]
    assert bad.size == 0, (f"{what}: {bad.size} codes differ, first at {bad[:4].tolist()}: "
                           f"{gpu.ravel()[bad[:4]].tolist()} vs {ref.ravel()[bad[:4]].tolist()}")


def compare_w(gpu: np.ndarray, ref: np.ndarray, what: str = "w") -> dict:
    g = gpu.astype(np.float64)
    r = ref.astype(np.float64)
    err = np.abs(g - r)
    ok = err <= W_RTOL * np.abs(r) + W_ATOL
    if not ok.all():
        i = int(np.argmax(err / (W_RTOL * np.abs(r) + W_ATOL)))
        raise AssertionError(f"{what}: {int((~ok).sum())} weights outside tolerance, max err "
                             f"{err.max():.3e}; worst at {i}: gpu {g[i]!r} ref {r[i]!r}")
    return {"w_max_rel": float((err / np.maximum(np.abs(r), 1e-30)).max())}


def s_condition(S: np.ndarray, k: np.ndarray, R: float = R_E4M3) -> tuple:
    """Sensitivity of ln S to relative changes of the group's max / min and to k.

    With S = max^k / 448 and (uncapped) k = ln R / ln R_X:
      d ln S = k [(1 - lam) d ln max + lam d ln min],   lam = ln max / ln R_X,
    and at fixed inputs d ln S = (k ln max) dk / k.  Derived from the oracle's
    own (S, k): k ln max = ln(448 S), ln R_X = ln R / k.
    """
    S = S.astype(np.float64)
    k = k.astype(np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        kln = np.where(S > 0, np.log(448.0 * np.where(S > 0, S, 1.0)), 0.0)
        lam = np.where(S > 0, kln / np.log(R), 0.0)  # = ln max / ln R_X
    kappa_state = k * (np.abs(1.0 - lam) + np.abs(lam))
    kappa_k = np.abs(kln)
    return kappa_state, kappa_k


def compare_meta(gpu_S, gpu_k, ref_S, ref_k, what: str, state_rel: float = STATE_REL) -> dict:
    gk = gpu_k.astype(np.float64)
    rk = ref_k.astype(np.float64)
    krel = np.abs(gk / rk - 1.0)
    assert krel.max() <= K_RTOL, f"{what}: k differs by {krel.max():.3e} relative"
    gS = gpu_S.astype(np.float64)
    rS = ref_S.astype(np.float64)
    zero = rS == 0
    assert np.array_equal(gS == 0, zero), f"{what}: zero scales differ"
    srel = np.zeros_like(rS)
    srel[~zero] = np.abs(gS[~zero] / rS[~zero] - 1.0)
    bad = srel > S_RTOL
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {srel.size} scales differ by more than "
                           f"{S_RTOL} relative; worst {srel.max():.3e}")
    return {"k_max_rel": float(krel.max()), "S_max_rel": float(srel.max()),
            "k_bit_equal_frac": float((gk == rk).mean()),
            "S_bit_equal_frac": float((gS == rS).mean())}


def adamw_like_state(n: int, G: int, seed: int, oracle):
    """A non-zero optimizer state coupled like real AdamW moments, quantized by the oracle.

    Per group a gradient scale s is drawn log-uniform in [1e-6, 1e-2]; per
    element s_e = s exp(0.5 z); then m ~ 0.23 s_e N(0, 1) (the spread of an
    EMA with beta1 = 0.9 of i.i.d. gradients) and v ~ s_e^2 (0.5 + U[0, 1]).
    Independent random codes would pair a large first moment with a tiny
    second moment, an update no AdamW trajectory produces.
    """
    import numpy as np
    from coat_fp8_adamw_gb300 import synth
    m, v = synth.adamw_like_moments_np(n, G, seed)
    mq, Sm, km = oracle.dre_quantize(m, G)
    vq, Sv, kv = oracle.dre_quantize(v, G)
    meta = np.stack([Sm, km, Sv, kv], axis=1).astype(np.float32)
    return mq, vq, np.ascontiguousarray(meta)
