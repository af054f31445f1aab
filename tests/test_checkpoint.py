"""Checkpoint and resume.  The library keeps no state between calls: the whole
optimizer state is the caller's flat buffers (w fp32, m and v E4M3 codes,
one (S_m, k_m, S_v, k_v) record per group).  A checkpoint is a raw save of
those bytes, and a run resumed from it must continue bit for bit as if it
had never stopped.  The step index t is the caller's too (it sets the bias
corrections) and is saved beside the buffers."""
import os

import numpy as np
import pytest

import coat_fp8_adamw_gb300 as coat
import oracle
from coat_fp8_adamw_gb300 import synth

HP = synth.HYPER
N, G = 128 * 96 + 40, 128          # a ragged last group
STEPS, STOP = 5, 2


def _grads(n, steps):
    rng = np.random.default_rng(21)
    return [synth.f32_to_bf16_bits((rng.standard_normal(n) * 1e-3).astype(np.float32))
            for _ in range(steps)]


def _initial(n, G):
    rng = np.random.default_rng(20)
    w = (rng.standard_normal(n) * 0.02).astype(np.float32)
    mq, vq, meta = synth.zero_state_np(n, G)
    return [w, mq, vq, meta]


def _save(path, state, t):
    for name, a in zip(("w", "mq", "vq", "meta"), state):
        a.tofile(os.path.join(path, name + ".bin"))
    with open(os.path.join(path, "step.txt"), "w") as fh:
        fh.write(str(t))


def _load(path, n, G):
    ng = (n + G - 1) // G
    w = np.fromfile(os.path.join(path, "w.bin"), np.float32)
    mq = np.fromfile(os.path.join(path, "mq.bin"), np.uint8)
    vq = np.fromfile(os.path.join(path, "vq.bin"), np.uint8)
    meta = np.fromfile(os.path.join(path, "meta.bin"), np.float32).reshape(ng, 4)
    with open(os.path.join(path, "step.txt")) as fh:
        t = int(fh.read())
    assert w.size == n and mq.size == n and vq.size == n
    return [w, mq, vq, meta], t


def _same(a, b):
    return all(np.array_equal(x.view(np.uint8), y.view(np.uint8)) for x, y in zip(a, b))


def _oracle_run(state, grads, t0, t1):
    for t in range(t0, t1 + 1):
        oracle.adamw_step(state[0], grads[t - 1], state[1], state[2], state[3], G, HP["beta1"],
                          HP["beta2"], HP["lr"], HP["eps"], HP["weight_decay"], t)
    return state


def test_oracle_run_resumes_bit_for_bit(tmp_path):
    grads = _grads(N, STEPS)
    straight = _oracle_run(_initial(N, G), grads, 1, STEPS)
    part = _oracle_run(_initial(N, G), grads, 1, STOP)
    _save(str(tmp_path), part, STOP)
    state, t = _load(str(tmp_path), N, G)
    resumed = _oracle_run(state, grads, t + 1, STEPS)
    assert _same(straight, resumed)


@pytest.mark.gpu
def test_device_step_resumes_bit_for_bit(tmp_path):
    import torch
    from coat_fp8_adamw_gb300 import _build
    _build.build()
    grads = _grads(N, STEPS)
    g_dev = [torch.from_numpy(g.view(np.int16)).cuda().view(torch.bfloat16) for g in grads]

    def run(state, t0, t1):
        d = [torch.from_numpy(a.copy()).cuda() for a in state]
        for t in range(t0, t1 + 1):
            coat.coat_fp8_adamw_step(d[0], g_dev[t - 1], d[1], d[2], d[3], G, HP["beta1"],
                                     HP["beta2"], HP["lr"], HP["eps"], HP["weight_decay"], t)
        torch.cuda.synchronize()
        return [x.cpu().numpy() for x in d]

    straight = run(_initial(N, G), 1, STEPS)
    part = run(_initial(N, G), 1, STOP)
    _save(str(tmp_path), part, STOP)
    state, t = _load(str(tmp_path), N, G)
    resumed = run(state, t + 1, STEPS)
    assert _same(straight, resumed)
    # the host-state step continues the same run from the same checkpoint
    state, t = _load(str(tmp_path), N, G)
    h = [torch.from_numpy(a.copy()).pin_memory() for a in state]
    ws = torch.empty(coat.coat_fp8_adamw_step_host_workspace_bytes(4096, G), dtype=torch.uint8,
                     device="cuda")
    for tt in range(t + 1, STEPS + 1):
        hg = torch.from_numpy(grads[tt - 1].view(np.int16)).view(torch.bfloat16).pin_memory()
        coat.coat_fp8_adamw_step_host(h[0], hg, h[1], h[2], h[3], G, HP["beta1"], HP["beta2"],
                                      HP["lr"], HP["eps"], HP["weight_decay"], tt, ws)
    assert _same(straight, [x.numpy() for x in h])
