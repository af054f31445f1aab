"""The step kernel on groups built around hard fp32 roundings of dequantized
moments, teacher-forced against the oracle.

A dequantized moment is the fp32 value of sign(q) (|E4M3(q)| S)^(1/k) (COAT
review page, section 3: the dequantized tensor is X_FP32).  Each group here
puts one such value, lying within 1e-5 ulp of an fp32 rounding midpoint, at
the group's smallest |m_t|, cancelled about 20-fold by the gradient:
m_t = beta1 prev + (1 - beta1) g with g close to -beta1 prev / (1 - beta1).
A one-ulp slip in prev is then about 20 ulps of the group minimum and moves
k_m by a few ulps, so k_m must equal the oracle's bit for bit.  The cases are
the recorded one from step 50 of the 4096 x 4096 trajectory
(tests/golden/hard_rounding_case.txt) and values found by a float64 search.
"""
import os

import numpy as np
import pytest
import torch

import _parity as P
import coat_fp8_adamw_gb300 as coat
import oracle
from coat_fp8_adamw_gb300 import synth

pytestmark = pytest.mark.gpu
HP = synth.HYPER
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _built():
    from coat_fp8_adamw_gb300 import _build
    _build.build()
    coat.lib()


def _recorded_case():
    with open(os.path.join(ROOT, "tests", "golden", "hard_rounding_case.txt")) as fh:
        line = [ln for ln in fh if not ln.startswith("#")][0]
    code, s, k, _, _ = (int(x) for x in line.split())
    return code & 0x7F, np.uint32(s).view(np.float32), np.uint32(k).view(np.float32)


def _searched_cases(count, seed):
    dec = oracle.e4m3_decode_all()
    rng = np.random.default_rng(seed)
    N = 4_000_000
    codes = rng.choice(np.arange(1, 0x7E, dtype=np.uint8), N)
    S = np.exp2(rng.uniform(-60.0, -2.0, N)).astype(np.float32)
    k = rng.uniform(1.05, 8.0, N).astype(np.float32)
    x = (np.abs(dec[codes]) * S.astype(np.float64)) ** (1.0 / k.astype(np.float64))
    ok = (x > 2.0 ** -120) & (x < 2.0 ** 100)
    frac = x / np.spacing(x.astype(np.float32)).astype(np.float64)
    dist = np.abs(frac - np.floor(frac) - 0.5)
    idx = np.nonzero(ok & (dist < 1e-5))[0][:count]
    return codes[idx], S[idx], k[idx]


def _groups(cases, G):
    """State and gradient of one group per case: element 0 holds the hard
    code, cancelled by its gradient; the other elements hold the largest code
    and a zero gradient (the group maximum).  Every second moment is stored as
    the largest code with k = 1 and S = P^2 / 448, P = (448 S_m)^(1/k_m) the
    largest first moment, so that v ~ m^2 as on an AdamW trajectory."""
    b1 = np.float32(HP["beta1"])
    n = len(cases) * G
    mq = np.full(n, 0x7E, np.uint8)
    vq = np.full(n, 0x7E, np.uint8)
    meta = np.zeros((len(cases), 4), np.float32)
    g = np.zeros(n, np.float32)
    for i, (code, S, k) in enumerate(cases):
        mq[i * G] = code
        pm = (448.0 * float(S)) ** (1.0 / float(k))
        meta[i] = (S, k, np.float32(pm * pm / 448.0), 1.0)
        prev = float(oracle.dre_dequantize(np.array([code], np.uint8), np.array([S]),
                                           np.array([k]), 1)[0])
        g[i * G] = -float(b1) * prev * 0.95 / (1.0 - float(b1))
    rng = np.random.default_rng(3)
    w = (rng.standard_normal(n) * 0.02).astype(np.float32)
    return w, synth.f32_to_bf16_bits(g), mq, vq, meta


def test_step_rounds_hard_dequantized_minima_exactly():
    G = 16
    c0 = _recorded_case()
    codes, S, k = _searched_cases(80, seed=91)
    assert codes.size >= 30
    cases = [c0] + list(zip(codes, S, k))
    w, g, mq, vq, meta = _groups(cases, G)
    t = 5
    d = [torch.from_numpy(x.copy()).cuda() for x in (w, mq, vq, meta)]
    gd = torch.from_numpy(g.view(np.int16)).cuda().view(torch.bfloat16)
    coat.coat_exact_recompute_counts(reset=True)
    coat.coat_fp8_adamw_step(d[0], gd, d[1], d[2], d[3], G, HP["beta1"], HP["beta2"], HP["lr"],
                             HP["eps"], HP["weight_decay"], t)
    dq, dk = coat.coat_exact_recompute_counts(reset=True)
    gw, gm, gv, gmeta = (x.cpu().numpy() for x in d)
    oracle.adamw_step(w, g, mq, vq, meta, G, HP["beta1"], HP["beta2"], HP["lr"], HP["eps"],
                      HP["weight_decay"], t)
    print("float64 recomputations: dequantized", dq, "k", dk, "of", len(cases), "hard cases")
    # the minima must be what the oracle has: k_m bit for bit
    bad = np.nonzero(gmeta[:, 1].view(np.uint32) != meta[:, 1].view(np.uint32))[0]
    assert bad.size == 0, [(int(i), float(gmeta[i, 1]), float(meta[i, 1])) for i in bad[:5]]
    P.compare_w(gw, w)
    P.compare_meta(gmeta[:, 0], gmeta[:, 1], meta[:, 0], meta[:, 1], "hard (S_m, k_m)")
    P.compare_meta(gmeta[:, 2], gmeta[:, 3], meta[:, 2], meta[:, 3], "hard (S_v, k_v)")
    d_m = np.abs(P.code_ordinal(gm) - P.code_ordinal(mq))
    assert d_m.max() <= 1
    assert dq >= 1, "the hard values must reach the float64 recomputation"
