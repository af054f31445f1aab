"""The step kernel's fast-path error bound and candidate windows, checked on a
float32 model with worst-case SFU errors.

The fused step evaluates every new moment on a fast float32 path (SFU exp2)
and re-evaluates exactly only the elements inside per-group windows around
the fast extremes; the windows rest on the bound
    |m_fast - m| <= eps_m T_j,   T_j = beta1 |prev_j| + (1 - beta1) |g_j|,
    |v_fast - v| <= eps_v v,
with eps = 2 E + 1.5e-7 + 1.25e-7 (17.81 / k + 1) and E the relative error
of the SFU exp2 (the kernel's constant, 2^-22, checked on the hardware by
test_gpu_sfu_bound.py).

This model repeats the fast path's float32 operations in numpy, in the
kernel's order, and gives every exp2 result a relative error of exactly
+2^-22, -2^-22 or a random one of the two -- the worst the bound allows,
where the hardware itself stays near 2^-22.7.  The exact moments come from
the oracle's dequantizer and the definition of the moment updates.  Checked:
the bound for every element, and that every group's exact extremes lie
inside the kernel's candidate windows built from the fast values.
"""
import numpy as np
import pytest

import oracle
from coat_fp8_adamw_gb300 import synth

import _parity as P
from _kernel_consts import kernel_ex2_bound

F = np.float32
KERNEL_EX2_ERR = kernel_ex2_bound()   # the SFU bound the kernel's fast_err budgets
E_SFU = KERNEL_EX2_ERR                # the SFU error the model injects
BETA1, BETA2 = F(synth.HYPER["beta1"]), F(synth.HYPER["beta2"])
OMB1 = F(1.0 - np.float64(BETA1))          # exact: 1 - beta is a float for beta in [0.5, 1)
OMB2 = F(1.0 - np.float64(BETA2))
DEC = oracle.e4m3_decode_all()
with np.errstate(divide="ignore"):
    L32 = np.where(np.arange(256) & 0x7F, np.log2(np.abs(DEC) / 448.0), -1e30).astype(F)


def fast_err(rk: np.ndarray) -> np.ndarray:
    return (F(2.0 * KERNEL_EX2_ERR) + F(1.5e-7) + F(1.25e-7) * (F(17.81) * rk + F(1.0))).astype(F)


def sfu_exp2(x: np.ndarray, sign: np.ndarray) -> np.ndarray:
    """2^x with a relative error of exactly sign * 2^-22, flushed below 2^-126."""
    y = np.exp2(x.astype(np.float64)) * (1.0 + sign * E_SFU)
    y = np.where(y < 2.0 ** -126, 0.0, y)
    return y.astype(F)


def fma32(a, b, c):
    # products of two floats are exact in float64; the float64 sum then rounds
    # at 2^-53, far below every margin checked here
    return (a.astype(np.float64) * b.astype(np.float64) + c.astype(np.float64)).astype(F)


def fast_params(S: np.ndarray, k: np.ndarray, sign: np.ndarray):
    """Per group: P = (448 S)^(1/k) (log2 in high precision, one SFU exp2 of the
    fractional part) and rk = float(1/k)."""
    rk = (1.0 / k.astype(np.float64)).astype(F)
    with np.errstate(divide="ignore"):
        z = (np.log2(448.0 * S.astype(np.float64)) / k.astype(np.float64))
    z = np.where(S > 0, z, 0.0)
    n = np.rint(z)
    frac = (z - n).astype(F)
    Pv = (sfu_exp2(frac, sign).astype(np.float64) * np.exp2(n)).astype(F)
    return np.where(S > 0, Pv, F(0)), rk


def model_step(mq, vq, meta, gf, G, rng, mode):
    """Fast m and v of the model, the exact ones, and T_j."""
    n = mq.size
    ng = n // G
    grp = np.repeat(np.arange(ng), G)

    def signs(size):
        if mode == "plus":
            return np.ones(size)
        if mode == "minus":
            return -np.ones(size)
        return rng.choice([-1.0, 1.0], size)

    Pm, rkm = fast_params(meta[:, 0], meta[:, 1], signs(ng))
    Pv, rkv = fast_params(meta[:, 2], meta[:, 3], signs(ng))
    em = sfu_exp2((L32[mq & 0x7F] * rkm[grp]).astype(F), signs(n))
    ev = sfu_exp2((L32[vq & 0x7F] * rkv[grp]).astype(F), signs(n))
    bPm = (BETA1 * Pm).astype(F)[grp]
    bPs = np.where(mq & 0x80, -bPm, bPm).astype(F)
    bPv = (BETA2 * Pv).astype(F)[grp]
    m_fast = fma32(bPs, em, (OMB1 * gf).astype(F))
    v_fast = fma32(bPv, ev, ((OMB2 * gf).astype(F) * gf).astype(F))
    # exact: the oracle's dequantized stored moments, then the EMA rounded once
    prev_m = oracle.dre_dequantize(mq, meta[:, 0], meta[:, 1], G).astype(np.float64)
    prev_v = oracle.dre_dequantize(vq, meta[:, 2], meta[:, 3], G).astype(np.float64)
    g64 = gf.astype(np.float64)
    m = (float(BETA1) * prev_m + float(OMB1) * g64).astype(F)
    v = (float(BETA2) * prev_v + float(OMB2) * g64 * g64).astype(F)
    Tj = float(BETA1) * np.abs(prev_m) + float(OMB1) * np.abs(g64)
    Tv = float(BETA2) * prev_v + float(OMB2) * g64 * g64
    return m_fast, v_fast, m, v, Tj, Tv, fast_err(rkm), fast_err(rkv), Pm


def check_windows(m_fast, v_fast, m, v, gf, eps_m, eps_v, Pm, G):
    """Every exact extreme of every group lies in the kernel's candidate windows."""
    ng = m.size // G
    mf, vf = m_fast.reshape(ng, G), v_fast.reshape(ng, G)
    me, ve = np.abs(m.reshape(ng, G)), v.reshape(ng, G)
    ag = np.abs(gf.reshape(ng, G))
    amf = np.abs(mf)
    fmx_m, fmx_v, gmx = amf.max(1), vf.max(1), ag.max(1)
    with np.errstate(invalid="ignore"):
        fmn_m = np.where(amf > 0, amf, np.inf).min(1)
        fmn_v = np.where(vf > 0, vf, np.inf).min(1)
    fmn_m = np.where(np.isfinite(fmn_m), fmn_m, 0).astype(F)
    fmn_v = np.where(np.isfinite(fmn_v), fmn_v, 0).astype(F)
    T = fma32(np.full(ng, BETA1), (Pm * (F(1) + eps_m)).astype(F), (OMB1 * gmx).astype(F))
    hi_m = (fmx_m - (F(2) * eps_m * T).astype(F)).astype(F)
    hi_v = (fmx_v * (F(1) - F(2) * eps_v)).astype(F)
    lo_v = np.where(fmn_v > 0, (fmn_v * (F(1) + F(4) * eps_v)).astype(F), F(-1))
    a0 = np.where(fmn_m > 0, fma32(eps_m, T, fmn_m), -np.inf)
    Tjf = fma32(np.full_like(amf, 2 * OMB1), ag, amf)
    lo_m = np.maximum(fma32(eps_m[:, None] * np.ones_like(amf), Tjf, np.broadcast_to(a0[:, None], amf.shape).astype(F)),
                      (F(1024) * eps_m)[:, None] * Tjf)
    live = (amf > 0) | (ag > 0)
    cand = [amf >= hi_m[:, None], (amf <= lo_m) & live, vf >= hi_v[:, None], vf <= lo_v[:, None]]
    nz_m, nz_v = me > 0, ve > 0
    mx_m = me == me.max(1, keepdims=True)
    mx_v = ve == ve.max(1, keepdims=True)
    mn_m = nz_m & (me == np.where(nz_m, me, np.inf).min(1, keepdims=True))
    mn_v = nz_v & (ve == np.where(nz_v, ve, np.inf).min(1, keepdims=True))
    for name, truth, c, has in (("max m", mx_m, cand[0], me.max(1) > 0),
                                ("min m", mn_m, cand[1], nz_m.any(1)),
                                ("max v", mx_v, cand[2], ve.max(1) > 0),
                                ("min v", mn_v, cand[3], nz_v.any(1))):
        # an extreme is found when at least one element attaining it is a candidate
        found = (truth & c).any(1)
        missed = has & ~found
        assert not missed.any(), f"{name}: {int(missed.sum())} groups' exact extreme outside the window"
    return [float(c.sum(1).mean()) for c in cand]


def adamw_like_case(seed, G=128, ng=2048):
    n = G * ng
    mq, vq, meta = P.adamw_like_state(n, G, seed, oracle)
    prev_v = oracle.dre_dequantize(vq, meta[:, 2], meta[:, 3], G).reshape(ng, G)
    scale = np.sqrt(prev_v.mean(1, dtype=np.float64) + 1e-30)
    rng = np.random.default_rng(seed + 100)
    g = rng.standard_normal((ng, G)) * scale[:, None] * np.exp(0.5 * rng.standard_normal((ng, G)))
    gbits = synth.f32_to_bf16_bits(g.astype(F).ravel())
    gf = synth.bf16_bits_to_f32(gbits)
    return mq, vq, meta, gf


@pytest.mark.parametrize("mode", ["plus", "minus", "random"])
@pytest.mark.parametrize("seed", [1, 2])
def test_bound_and_windows_hold_with_worst_case_sfu_errors(mode, seed):
    G = 128
    mq, vq, meta, gf = adamw_like_case(seed, G)
    rng = np.random.default_rng(seed)
    m_fast, v_fast, m, v, Tj, Tv, eps_m, eps_v, Pm = model_step(mq, vq, meta, gf, G, rng, mode)
    grp = np.repeat(np.arange(m.size // G), G)
    err_m = np.abs(m_fast.astype(np.float64) - m)
    err_v = np.abs(v_fast.astype(np.float64) - v)
    ratio_m = err_m / np.maximum(eps_m[grp] * Tj, 1e-300)
    ratio_v = err_v / np.maximum(eps_v[grp] * Tv, 1e-300)
    assert ratio_m.max() <= 1.0, f"m: error reaches {ratio_m.max():.3f} of the bound"
    assert ratio_v.max() <= 1.0, f"v: error reaches {ratio_v.max():.3f} of the bound"
    check_windows(m_fast, v_fast, m, v, gf, eps_m, eps_v, Pm, G)


@pytest.mark.parametrize("G", [16, 32, 256])
def test_windows_hold_for_other_group_sizes(G):
    mq, vq, meta, gf = adamw_like_case(7 + G, G, ng=8192 // (G // 16))
    rng = np.random.default_rng(G)
    m_fast, v_fast, m, v, Tj, Tv, eps_m, eps_v, Pm = model_step(mq, vq, meta, gf, G, rng, "random")
    check_windows(m_fast, v_fast, m, v, gf, eps_m, eps_v, Pm, G)


def test_the_model_detects_a_bound_that_is_too_tight():
    """With an SFU error four times what the bound budgets, the model reports
    the violation: the check is not vacuous."""
    global E_SFU
    G = 128
    mq, vq, meta, gf = adamw_like_case(3, G, ng=512)
    saved = E_SFU
    try:
        E_SFU = 2.0 ** -20
        m_fast, v_fast, m, v, Tj, Tv, eps_m, eps_v, Pm = model_step(
            mq, vq, meta, gf, G, np.random.default_rng(0), "plus")
    finally:
        E_SFU = saved
    grp = np.repeat(np.arange(m.size // G), G)
    ratio_v = np.abs(v_fast.astype(np.float64) - v) / np.maximum(eps_v[grp] * Tv, 1e-300)
    assert ratio_v.max() > 1.0
