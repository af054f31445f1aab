"""The library's step on a data-parallel shard layout, on one GPU.

Each rank's pieces of the bucket-interleaved, zero-padded layout are stepped
by their own launches (the ranks are independent: no launch waits on another)
and the reassembled state must equal one launch over the whole unpadded
buffer bit for bit, and the oracle within the parity tolerances.  A world-1
NCCL process group then runs the asynchronous reduce-scatter / wait / step
orchestration on the GPU's streams.
"""
import os
import socket

import numpy as np
import pytest
import torch

import _parity as P
import coat_fp8_adamw_gb300 as coat
import oracle
from coat_fp8_adamw_gb300 import synth
from coat_fp8_adamw_gb300.shard import ShardLayout, from_locals, sharded_step, to_local

pytestmark = pytest.mark.gpu
HP = synth.HYPER
ARGS = (HP["beta1"], HP["beta2"], HP["lr"], HP["eps"], HP["weight_decay"])


@pytest.fixture(scope="module", autouse=True)
def _built():
    from coat_fp8_adamw_gb300 import _build
    _build.build()
    coat.lib()


def _state(n, G, seed):
    rng = np.random.default_rng(seed)
    w = (rng.standard_normal(n) * 0.02).astype(np.float32)
    mq, vq, meta = P.adamw_like_state(n, G, seed, oracle)
    return w, mq, vq, meta


def _grad(n, seed):
    rng = np.random.default_rng(seed)
    return synth.f32_to_bf16_bits((rng.standard_normal(n) * 10.0 ** rng.uniform(-5, -2, n)).astype(np.float32))


def _pad(a, length, fill):
    out = np.empty((length,) + a.shape[1:], a.dtype)
    out[:] = fill
    out[:a.shape[0]] = a
    return torch.from_numpy(out).cuda()


@pytest.mark.parametrize("G,world,buckets", [(128, 3, 2), (16, 8, 3), (4, 2, 5), (256, 5, 1)])
def test_pieces_match_one_launch(G, world, buckets):
    n = 3 * 65536 + 4321
    L = ShardLayout(n, G, world, buckets)
    w, mq, vq, meta = _state(n, G, G + world)
    ng = meta.shape[0]
    # one launch over the whole unpadded state, two steps
    full = [torch.from_numpy(a.copy()).cuda() for a in (w, mq, vq, meta)]
    # the padded layout, each rank's pieces stepped by their own launches
    pw, pm, pv = _pad(w, L.padded, 0), _pad(mq, L.padded, 0), _pad(vq, L.padded, 0)
    pmeta = _pad(meta, L.padded // G, np.array([0, 1, 0, 1], np.float32))
    loc = [[to_local(x, L, r) for x in (pw, pm, pv)] + [to_local(pmeta, L, r, per_group=True)]
           for r in range(world)]
    gs = []
    for t in (1, 2):
        g = _grad(n, 10 * t + G)
        gs.append(g)
        gd = torch.from_numpy(g.view(np.int16)).cuda().view(torch.bfloat16)
        coat.coat_fp8_adamw_step(full[0], gd, full[1], full[2], full[3], G, *ARGS, t)
        gpad = torch.zeros(L.padded, dtype=torch.bfloat16, device="cuda")
        gpad[:n] = gd
        for r in range(world):
            gl = to_local(gpad, L, r)
            wl, ml, vl, metal = loc[r]
            for b in range(buckets):
                s = L.local_piece(b)
                coat.coat_fp8_adamw_step(wl[s], gl[s], ml[s], vl[s], metal[L.groups(s)], G, *ARGS, t)
        if t == 1:
            first = [from_locals([loc[r][i] for r in range(world)], L, per_group=(i == 3)).cpu().numpy()
                     for i in range(4)]
    torch.cuda.synchronize()
    got = [from_locals([loc[r][i] for r in range(world)], L, per_group=(i == 3)) for i in range(4)]
    for i, name in enumerate(("w", "m_q", "v_q", "meta")):
        a = got[i][:n if i < 3 else ng].contiguous().cpu().numpy()
        b = full[i].cpu().numpy()
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8)), f"{name} differs from one launch"
    assert not got[0][n:].any() and not got[1][n:].any() and not got[2][n:].any()
    pad_meta = got[3][ng:].cpu()
    assert torch.all(pad_meta == torch.tensor([0.0, 1.0, 0.0, 1.0]))
    # the first step against the oracle
    ref = [a.copy() for a in (w, mq, vq, meta)]
    oracle.adamw_step(ref[0], gs[0], ref[1], ref[2], ref[3], G, *ARGS, 1)
    P.compare_w(first[0][:n], ref[0], "sharded w")
    P.compare_codes(first[1][:n], ref[1], "sharded m codes")
    P.compare_codes(first[2][:n], ref[2], "sharded v codes")
    fm = first[3][:ng]
    P.compare_meta(fm[:, 0], fm[:, 1], ref[3][:, 0], ref[3][:, 1], "sharded (S_m, k_m)")
    P.compare_meta(fm[:, 2], fm[:, 3], ref[3][:, 2], ref[3][:, 3], "sharded (S_v, k_v)")


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def test_nccl_world_one_orchestration():
    import torch.distributed as dist
    if not dist.is_nccl_available():
        pytest.skip("torch.distributed has no NCCL backend")
    G, n, buckets = 128, 2 * 65536 + 999, 4
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(_free_port()))
    dist.init_process_group("nccl", rank=0, world_size=1, device_id=torch.device("cuda:0"))
    try:
        L = ShardLayout(n, G, 1, buckets)
        w, mq, vq, meta = _state(n, G, 77)
        g = _grad(n, 78)
        gd = torch.from_numpy(g.view(np.int16)).cuda().view(torch.bfloat16)
        full = [torch.from_numpy(a.copy()).cuda() for a in (w, mq, vq, meta)]
        coat.coat_fp8_adamw_step(full[0], gd, full[1], full[2], full[3], G, *ARGS, 1)
        pw, pm, pv = _pad(w, L.padded, 0), _pad(mq, L.padded, 0), _pad(vq, L.padded, 0)
        pmeta = _pad(meta, L.padded // G, np.array([0, 1, 0, 1], np.float32))
        gpad = torch.zeros(L.padded, dtype=torch.bfloat16, device="cuda")
        gpad[:n] = gd
        gloc = torch.empty(L.local, dtype=torch.bfloat16, device="cuda")
        sharded_step(coat.coat_fp8_adamw_step, L, 0, pw, pm, pv, pmeta, gpad, gloc, *ARGS, 1)
        torch.cuda.synchronize()
        assert torch.equal(gloc, gpad)
        for a, b in ((pw[:n], full[0]), (pm[:n], full[1]), (pv[:n], full[2]),
                     (pmeta[:full[3].shape[0]], full[3])):
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    finally:
        dist.destroy_process_group()
