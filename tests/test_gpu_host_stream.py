"""coat_fp8_adamw_step_host: the step over a host-resident state, streamed
through a device workspace, equals the device step bit for bit."""
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


def _state(n, G, seed):
    rng = np.random.default_rng(seed)
    w = (rng.standard_normal(n) * 0.02).astype(np.float32)
    g = synth.f32_to_bf16_bits((rng.standard_normal(n) * 1e-3).astype(np.float32))
    mq, vq, meta = P.adamw_like_state(n, G, seed, oracle)
    return w, g, mq, vq, meta


def _device_step(w, g, mq, vq, meta, G, t):
    d = [torch.from_numpy(x.copy()).cuda() for x in (w, mq, vq, meta)]
    gd = torch.from_numpy(g.view(np.int16)).cuda().view(torch.bfloat16)
    coat.coat_fp8_adamw_step(d[0], gd, d[1], d[2], d[3], G, HP["beta1"], HP["beta2"], HP["lr"],
                             HP["eps"], HP["weight_decay"], t)
    torch.cuda.synchronize()
    return [x.cpu().numpy() for x in d]


def _host_step(w, g, mq, vq, meta, G, t, ws_bytes, pinned=True):
    h = [torch.from_numpy(x.copy()) for x in (w, mq, vq, meta)]
    hg = torch.from_numpy(g.view(np.int16).copy()).view(torch.bfloat16)
    if pinned:
        h = [x.pin_memory() for x in h]
        hg = hg.pin_memory()
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    coat.coat_fp8_adamw_step_host(h[0], hg, h[1], h[2], h[3], G, HP["beta1"], HP["beta2"],
                                  HP["lr"], HP["eps"], HP["weight_decay"], t, ws)
    return [x.numpy() for x in h]


@pytest.mark.parametrize("n,G,chunk,pinned", [(50_000 + 13, 128, 4096, True),
                                              (200_000, 16, 8192, True),
                                              (70_000 + 1, 256, 1 << 20, False),
                                              (4096 * 5, 64, 4096, True)])
def test_host_stream_matches_device_step(n, G, chunk, pinned):
    w, g, mq, vq, meta = _state(n, G, n % 1000 + G)
    ws_bytes = coat.coat_fp8_adamw_step_host_workspace_bytes(chunk, G)
    assert ws_bytes > 0
    a = _device_step(w, g, mq, vq, meta, G, 5)
    b = _host_step(w, g, mq, vq, meta, G, 5, ws_bytes, pinned)
    for x, y in zip(a, b):
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8))


def test_host_stream_errors():
    n, G = 8192, 128
    w, g, mq, vq, meta = _state(n, G, 3)
    L = coat.lib()
    hw = torch.from_numpy(w.copy()).pin_memory()
    hg = torch.from_numpy(g.view(np.int16).copy()).pin_memory()
    hm = torch.from_numpy(mq.copy()).pin_memory()
    hv = torch.from_numpy(vq.copy()).pin_memory()
    hmeta = torch.from_numpy(meta.copy()).pin_memory()
    ws = torch.empty(coat.coat_fp8_adamw_step_host_workspace_bytes(4096, G), dtype=torch.uint8,
                     device="cuda")
    args = [hw.data_ptr(), hg.data_ptr(), hm.data_ptr(), hv.data_ptr(), hmeta.data_ptr(), n, G,
            0.9, 0.95, 1e-4, 1e-8, 0.1, 1]
    # workspace too small for one 4096-parameter chunk
    assert L.coat_fp8_adamw_step_host(*args, ws.data_ptr(), 1000, None) == 1
    # workspace in host memory
    hws = torch.empty(1 << 20, dtype=torch.uint8).pin_memory()
    assert L.coat_fp8_adamw_step_host(*args, hws.data_ptr(), 1 << 20, None) == 5
    # state in device memory
    dw = torch.from_numpy(w.copy()).cuda()
    bad = list(args)
    bad[0] = dw.data_ptr()
    assert L.coat_fp8_adamw_step_host(*bad, ws.data_ptr(), ws.numel(), None) == 1
    # misaligned workspace
    assert L.coat_fp8_adamw_step_host(*args, ws.data_ptr() + 16, ws.numel() - 16, None) == 2
    assert coat.coat_fp8_adamw_step_host_workspace_bytes(4096, 3) == 0
    torch.cuda.synchronize()
