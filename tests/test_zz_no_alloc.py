"""The step on host buffers through the library's static scratch
(coat_fp8_adamw_step_host_static, which allocates no device memory) against
the device-buffer step, through the C ABI.

The file name sorts last so that it runs after every other test (the scratch
is set up on first use, and must work whether or not other calls came
first); it also passes on its own in a fresh process.
"""
import numpy as np
import pytest
import torch

import _parity as P
import coat_fp8_adamw_gb300 as coat
import oracle
from coat_fp8_adamw_gb300 import synth

pytestmark = pytest.mark.gpu
HP = synth.HYPER


@pytest.fixture(scope="module", autouse=True)
def _built():
    from coat_fp8_adamw_gb300 import _build
    _build.build()
    coat.lib()


def _device_step(w, g, mq, vq, meta, G, t):
    d = [torch.from_numpy(x.copy()).cuda() for x in (w, mq, vq, meta)]
    gd = torch.from_numpy(g.view(np.int16)).cuda().view(torch.bfloat16)
    coat.coat_fp8_adamw_step(d[0], gd, d[1], d[2], d[3], G, HP["beta1"], HP["beta2"], HP["lr"],
                             HP["eps"], HP["weight_decay"], t)
    torch.cuda.synchronize()
    return [x.cpu().numpy() for x in d]


def _host(a, pinned):
    t = torch.from_numpy(np.ascontiguousarray(a).copy())
    return t.pin_memory() if pinned else t


def _check(host, ref, label):
    P.compare_w(host[0], ref[0], f"{label} w")
    P.compare_codes(host[1], ref[1], f"{label} m codes")
    P.compare_codes(host[2], ref[2], f"{label} v codes")
    P.compare_meta(host[3][:, 0], host[3][:, 1], ref[3][:, 0], ref[3][:, 1], f"{label} (S_m, k_m)")
    P.compare_meta(host[3][:, 2], host[3][:, 3], ref[3][:, 2], ref[3][:, 3], f"{label} (S_v, k_v)")
    # the same kernel on the same chunk-aligned tiles: identical results
    for a, b in zip(host, ref):
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8)), label


@pytest.mark.parametrize("G,n,chunk,pinned", [
    (128, 5 * 8192 + 1234, 8192, True),      # several chunks and a ragged tail
    (1, 3 * 4096 + 7, 4096, False),          # smallest chunk, pageable buffers
    (256, 2_500_000, 0, True),               # the default (largest) chunk, two chunks
])
def test_static_scratch_step_two_calls(G, n, chunk, pinned):
    rng = np.random.default_rng(G + n)
    w = (rng.standard_normal(n) * 0.02).astype(np.float32)
    mq, vq, meta = P.adamw_like_state(n, G, 7 + G, oracle)
    hw, hmq, hvq, hmeta = (_host(a, pinned) for a in (w, mq, vq, meta))
    state = [w, mq, vq, meta]
    for t in (5, 6):                          # two calls in a row on the same buffers
        g = synth.f32_to_bf16_bits((rng.standard_normal(n) * 1e-3).astype(np.float32))
        hg = _host(g.view(np.int16), pinned).view(torch.bfloat16)
        ref = _device_step(*state[:1], g, *state[1:], G, t)
        coat.coat_fp8_adamw_step_host_static(hw, hg, hmq, hvq, hmeta, G, HP["beta1"], HP["beta2"],
                                             HP["lr"], HP["eps"], HP["weight_decay"], t,
                                             chunk_params=chunk)
        host = [x.numpy().copy() for x in (hw, hmq, hvq, hmeta)]
        _check(host, ref, f"static G={G} n={n} t={t}")
        state = ref


def test_static_scratch_rejects_oversized_chunk():
    n, G = 4096, 128
    w = torch.zeros(n, dtype=torch.float32)
    g = torch.zeros(n, dtype=torch.bfloat16)
    mq = torch.zeros(n, dtype=torch.uint8)
    vq = torch.zeros(n, dtype=torch.uint8)
    meta = torch.zeros(n // G, 4, dtype=torch.float32)
    with pytest.raises(coat.CoatError) as ei:
        coat.coat_fp8_adamw_step_host_static(w, g, mq, vq, meta, G, 0.9, 0.95, 1e-4, 1e-8, 0.0, 1,
                                             chunk_params=coat.STATIC_SCRATCH_BYTES)
    assert ei.value.status == 6
    assert not w.any() and not mq.any()       # nothing ran
