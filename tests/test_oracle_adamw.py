"""Pins for the oracle's fused AdamW + DRE step (CPU only).

The AdamW update (COAT paper-review page, section 3, AdamW update rule) is
pinned, through the full quantized state path, against:

* the scalar closed form under a constant gradient: with m_0 = v_0 = 0 the
  bias-corrected moments are exactly g and g^2, so
  w_T = (1 - lr wd)^T w_0 - lr g/(|g| + eps) * sum_{j<T} (1 - lr wd)^j;
* torch.optim.AdamW in float64 (a library routine), in the cases where FP8
  storage is lossless: group size 1, and groups holding one non-zero
  element (R_X = 1, so k = 1 and the element maps to +-448);
* one step from the zero state at G = 128 (the state does not enter the
  first update), and the multi-step trajectory staying near unquantized
  AdamW, which catches a wrong un-expansion exponent.
"""
import numpy as np
import pytest
import torch

import oracle
from coat_fp8_adamw_gb300 import synth

HP = synth.HYPER


def _f32(x):
    return float(np.float32(x))


def _zero_state(n, G):
    return synth.zero_state_np(n, G)


def _run_oracle(w0, grads, G, hp=HP):
    n = w0.size
    w = w0.copy()
    mq, vq, meta = _zero_state(n, G)
    for t, g in enumerate(grads, start=1):
        oracle.adamw_step(w, g, mq, vq, meta, G, hp["beta1"], hp["beta2"], hp["lr"], hp["eps"],
                          hp["weight_decay"], t)
    return w, mq, vq, meta


def _torch_adamw(w0, grads_f32, hp=HP):
    p = torch.nn.Parameter(torch.from_numpy(w0.astype(np.float64)))
    opt = torch.optim.AdamW([p], lr=_f32(hp["lr"]), betas=(_f32(hp["beta1"]), _f32(hp["beta2"])),
                            eps=_f32(hp["eps"]), weight_decay=_f32(hp["weight_decay"]),
                            foreach=False)
    for g in grads_f32:
        p.grad = torch.from_numpy(g.astype(np.float64))
        opt.step()
    return p.detach().numpy()


def test_closed_form_constant_gradient():
    T = 25
    gvals = np.array([1e-3, -2.5e-3, 3e-8, -1e-8, 0.0, 0.5, -7.0, 1e-5], dtype=np.float32)
    gbits = synth.f32_to_bf16_bits(gvals)
    gexact = synth.bf16_bits_to_f32(gbits).astype(np.float64)
    w0 = np.array([0.02, -0.013, 0.5, -1.0, 0.7, 0.0, 1e-3, -3e-4], dtype=np.float32)
    w, _, _, _ = _run_oracle(w0, [gbits] * T, G=1)
    lr, wd, eps = _f32(HP["lr"]), _f32(HP["weight_decay"]), _f32(HP["eps"])
    decay = 1.0 - lr * wd
    geo = sum(decay ** j for j in range(T))
    want = decay ** T * w0.astype(np.float64) - lr * gexact / (np.abs(gexact) + eps) * geo
    assert np.allclose(w, want, rtol=2e-6, atol=1e-9)
    # the accumulated update itself is reproduced, not just the decay of w_0; each
    # step rounds w to fp32, which bounds the error by T half-ulps of |w|
    upd = w.astype(np.float64) - decay ** T * w0
    bound = 1e-5 * np.abs(want - decay ** T * w0) + T * np.abs(w0) * 2.0 ** -24 + 1e-12
    assert np.all(np.abs(upd - (want - decay ** T * w0)) <= bound)


def test_group_size_one_matches_torch_adamw():
    rng = np.random.default_rng(3)
    n, T = 512, 12
    w0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    grads = []
    for _ in range(T):
        g = (rng.standard_normal(n) * 10.0 ** rng.uniform(-6, -1, n)).astype(np.float32)
        grads.append(synth.f32_to_bf16_bits(g))
    w, _, _, _ = _run_oracle(w0, grads, G=1)
    ref = _torch_adamw(w0, [synth.bf16_bits_to_f32(g) for g in grads])
    assert np.allclose(w, ref, rtol=1e-6, atol=1e-9)


def test_single_nonzero_groups_match_torch_adamw():
    rng = np.random.default_rng(4)
    G, ngroups, T = 128, 16, 8
    n = G * ngroups
    w0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    pos = rng.integers(0, G, ngroups) + G * np.arange(ngroups)
    grads = []
    for _ in range(T):
        g = np.zeros(n, dtype=np.float32)
        g[pos] = rng.standard_normal(ngroups) * 1e-3
        grads.append(synth.f32_to_bf16_bits(g))
    w, mq, vq, meta = _run_oracle(w0, grads, G=G)
    ref = _torch_adamw(w0, [synth.bf16_bits_to_f32(g) for g in grads])
    assert np.allclose(w, ref, rtol=1e-6, atol=1e-9)
    # the one non-zero element of each group sits at +-448, everything else at 0
    assert np.all((mq[pos] & 0x7F) == 0x7E) and np.all(vq[pos] == 0x7E)
    others = np.ones(n, bool)
    others[pos] = False
    assert np.all(mq[others] == 0) and np.all(vq[others] == 0)
    assert np.all(meta[:, 1] == 1.0) and np.all(meta[:, 3] == 1.0)


def test_first_step_from_zero_state_is_textbook():
    wl = synth.workload("tiny")
    w0 = synth.init_weights_np(wl)
    g = synth.grad_np(wl, 1)
    w, mq, vq, meta = _run_oracle(w0, [g], G=wl.G)
    gf = synth.bf16_bits_to_f32(g).astype(np.float64)
    lr, wd, eps = _f32(HP["lr"]), _f32(HP["weight_decay"]), _f32(HP["eps"])
    want = w0 - lr * (gf / (np.abs(gf) + eps) + wd * w0)
    assert np.allclose(w, want, rtol=1e-6, atol=1e-9)
    # group 30 saw only zero gradients: zero state, S = 0, k = 1
    assert np.all(mq[30 * 128:31 * 128] == 0) and meta[30, 0] == 0 and meta[30, 1] == 1
    # the stored first moment dequantizes to (1 - beta1) g within the E4M3 grid error:
    # a normal code c holds the values y with |y - c| <= c/16, so c/y lies in
    # [16/17, 16/15] and the un-expanded value is within (16/15)^(1/k) - 1;
    # subnormal codes hold |y - c| <= 2^-10
    mdq = oracle.dre_dequantize(mq, meta[:, 0].copy(), meta[:, 1].copy(), wl.G).astype(np.float64)
    m1 = np.float32(1.0 - np.float32(HP["beta1"])) * gf
    k = np.repeat(meta[:, 1].astype(np.float64), wl.G)
    S = np.repeat(meta[:, 0].astype(np.float64), wl.G)
    normal = (mq & 0x7F) >= 0x08
    nz = m1 != 0
    rel = np.abs(mdq - m1) / np.where(nz, np.abs(m1), 1.0)
    assert np.all(rel[normal & nz] <= (16 / 15) ** (1 / k[normal & nz]) - 1 + 1e-6)
    sub = ~normal & nz
    y_true = np.abs(m1[sub]) ** k[sub] / S[sub]
    y_code = np.abs(mdq[sub]) ** k[sub] / S[sub]
    assert np.all(np.abs(y_true - y_code) <= 2.0 ** -10 * (1 + 1e-5))
    assert sub.sum() > 0 and normal.sum() > 3000


def test_quantized_trajectory_stays_near_unquantized_adamw():
    wl = synth.workload("tiny")
    w0 = synth.init_weights_np(wl)
    grads = [synth.grad_np(wl, t) for t in range(1, 11)]
    w, _, _, _ = _run_oracle(w0, grads, G=wl.G)
    ref = _torch_adamw(w0, [synth.bf16_bits_to_f32(g) for g in grads])
    step_sum = 10 * _f32(HP["lr"])
    assert np.max(np.abs(w - ref)) < 0.2 * step_sum
    # ...and is not trivially equal to it (the FP8 state is lossy)
    assert np.max(np.abs(w - ref)) > 1e-9


def test_zero_gradient_everywhere_only_decays():
    n, G = 300, 64  # ragged last group
    w0 = np.linspace(-1, 1, n).astype(np.float32)
    g = np.zeros(n, np.uint16)
    w, mq, vq, meta = _run_oracle(w0, [g] * 3, G=G)
    decay = 1.0 - _f32(HP["lr"]) * _f32(HP["weight_decay"])
    assert np.allclose(w, w0 * decay ** 3, rtol=1e-6, atol=1e-12)
    assert not mq.any() and not vq.any()
    assert np.all(meta[:, 0] == 0) and np.all(meta[:, 2] == 0)


def test_bad_arguments_are_rejected():
    w = np.zeros(4, np.float32)
    g = np.zeros(4, np.uint16)
    mq, vq, meta = _zero_state(4, 2)
    with pytest.raises(ValueError):
        oracle.adamw_step(w, g, mq, vq, meta, 2, 0.9, 0.95, 1e-4, 1e-8, 0.1, 0)
