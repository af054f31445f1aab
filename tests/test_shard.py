"""The data-parallel sharded step on the CPU: the group-aligned bucket layout,
and two gloo ranks that reduce-scatter their gradients and step their own
slices, against one oracle step over the whole unpadded state.

The step here is the oracle (a CPU stand-in for the library's kernel, which the
GPU test of the same layout runs); what is under test is the layout, the
padding and the collective orchestration of ``coat_fp8_adamw_gb300.shard``.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import _parity as P
import oracle
from coat_fp8_adamw_gb300 import synth
from coat_fp8_adamw_gb300.shard import ShardLayout, from_locals, to_local

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HP = synth.HYPER


@pytest.mark.parametrize("G", [1, 4, 16, 128, 256])
@pytest.mark.parametrize("world", [1, 2, 3, 8])
@pytest.mark.parametrize("buckets", [1, 2, 5])
def test_layout_partitions_the_padded_buffer(G, world, buckets):
    for n in (1, 15, 16, 17, G, G + 1, 4096, 12345, 1 << 20):
        L = ShardLayout(n, G, world, buckets)
        assert L.cap % L.unit == 0 and L.cap % G == 0 and L.cap % 16 == 0
        assert L.padded >= n and L.padded - n < buckets * world * L.unit + buckets * world
        cover = np.zeros(L.padded, np.int32)
        for b in range(buckets):
            bk = L.bucket(b)
            for r in range(world):
                p = L.piece(r, b)
                assert bk.start <= p.start and p.stop <= bk.stop
                assert p.start % L.unit == 0
                cover[p] += 1
                lp = L.local_piece(b)
                assert lp.stop - lp.start == p.stop - p.start
                assert L.real(r, b) == max(0, min(p.stop, n) - p.start)
        assert np.all(cover == 1)
        assert sum(L.real(r, b) for r in range(world) for b in range(buckets)) == n


def test_layout_rejects_bad_arguments():
    for args in ((0, 128, 2), (10, 128, 0), (10, 3, 2), (10, 512, 2)):
        with pytest.raises(ValueError):
            ShardLayout(*args)


def test_local_round_trip():
    L = ShardLayout(1000, 16, 3, 2)
    x = torch.arange(L.padded, dtype=torch.float32)
    meta = torch.arange(L.padded // 16 * 4, dtype=torch.float32).reshape(-1, 4)
    locs = [to_local(x, L, r) for r in range(3)]
    metas = [to_local(meta, L, r, per_group=True) for r in range(3)]
    assert all(t.numel() == L.local for t in locs)
    assert torch.equal(from_locals(locs, L), x)
    assert torch.equal(from_locals(metas, L, per_group=True), meta)
    # rank 1's second piece starts at bucket 1's start plus one piece
    assert locs[1][L.cap].item() == 1 * 3 * L.cap + L.cap


def _oracle_step(w, g, m_q, v_q, meta, G, beta1, beta2, lr, eps, wd, t):
    """The step callable of the sharded orchestration, on CPU tensor views."""
    oracle.adamw_step(w.numpy(), g.view(torch.int16).numpy().view(np.uint16), m_q.numpy(),
                      v_q.numpy(), meta.numpy(), G, beta1, beta2, lr, eps, wd, t, nthreads=1)


CASES = [(5077, 128, 3), (3001, 4, 2), (700, 16, 1)]


def _padded_state(n, G, L, seed):
    rng = np.random.default_rng(seed)
    w = np.zeros(L.padded, np.float32)
    w[:n] = rng.standard_normal(n) * 0.02
    mq = np.zeros(L.padded, np.uint8)
    vq = np.zeros(L.padded, np.uint8)
    meta = np.tile(np.array([0, 1, 0, 1], np.float32), (L.padded // G, 1))
    mq[:n], vq[:n], meta[:(n + G - 1) // G] = P.adamw_like_state(n, G, seed, oracle)
    return w, mq, vq, meta


def _local_grad(n, L, seed):
    rng = np.random.default_rng(seed)
    g = np.zeros(L.padded, np.float32)
    g[:n] = rng.standard_normal(n) * 10.0 ** rng.uniform(-5, -2, n)
    return torch.from_numpy(synth.f32_to_bf16_bits(g).view(np.int16)).view(torch.bfloat16)


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import torch.distributed as dist
    from coat_fp8_adamw_gb300.shard import all_gather_padded, sharded_step
    dist.init_process_group("gloo", rank=rank, world_size=world)
    res = {}
    for n, G, buckets in CASES:
        L = ShardLayout(n, G, world, buckets)
        w, mq, vq, meta = (torch.from_numpy(a) for a in _padded_state(n, G, L, n))
        wl, ml, vl = to_local(w, L, rank), to_local(mq, L, rank), to_local(vq, L, rank)
        metal = to_local(meta, L, rank, per_group=True)
        g_pad = _local_grad(n, L, 1000 * rank + n)
        g_loc = torch.empty(L.local, dtype=torch.bfloat16)
        for t in (1, 2):                    # two steps: the second starts from a sharded state
            sharded_step(_oracle_step, L, rank, wl, ml, vl, metal, g_pad, g_loc, HP["beta1"],
                         HP["beta2"], HP["lr"], HP["eps"], HP["weight_decay"], t)
            if t == 1:
                g_red1 = all_gather_padded(g_loc, L).view(torch.int16)
        res[(n, G, buckets)] = tuple(x.numpy().copy() for x in (
            g_red1, all_gather_padded(g_loc, L).view(torch.int16), all_gather_padded(wl, L),
            all_gather_padded(ml, L), all_gather_padded(vl, L),
            all_gather_padded(metal, L, per_group=True)))
    out[rank] = res
    dist.barrier()
    dist.destroy_process_group()


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def test_two_ranks_match_one_unsharded_step():
    oracle.build()
    world = 2
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(300)
        assert p.exitcode == 0
    for n, G, buckets in CASES:
        L = ShardLayout(n, G, world, buckets)
        r0, r1 = out[0][(n, G, buckets)], out[1][(n, G, buckets)]
        for a, b in zip(r0, r1):
            assert np.array_equal(a.view(np.uint8), b.view(np.uint8)), "ranks gather the same state"
        g_red1, g_red2, w_sh, m_sh, v_sh, meta_sh = r0
        # the reduce-scatter delivered the bf16 sum of both ranks' gradients
        g0 = _local_grad(n, L, n).float()
        g1 = _local_grad(n, L, 1000 + n).float()
        expect = (g0 + g1).bfloat16().view(torch.int16).numpy()
        assert np.array_equal(g_red1.view(np.int16), expect)
        assert np.array_equal(g_red2.view(np.int16), expect)
        # one unsharded oracle step per step on the first n elements
        w, mq, vq, meta = _padded_state(n, G, L, n)
        ng = (n + G - 1) // G
        w, mq, vq, meta = w[:n].copy(), mq[:n].copy(), vq[:n].copy(), meta[:ng].copy()
        gb = np.ascontiguousarray(g_red1.view(np.uint16)[:n])
        for t in (1, 2):
            oracle.adamw_step(w, gb, mq, vq, meta, G, HP["beta1"], HP["beta2"], HP["lr"],
                              HP["eps"], HP["weight_decay"], t)
        assert np.array_equal(w_sh[:n].view(np.uint32), w.view(np.uint32))
        assert np.array_equal(m_sh[:n], mq) and np.array_equal(v_sh[:n], vq)
        assert np.array_equal(meta_sh[:ng].view(np.uint32), meta.view(np.uint32))
        # padding stays zero with its records at the initial (0, 1) pair
        assert not w_sh[n:].any() and not m_sh[n:].any() and not v_sh[n:].any()
        assert np.all(meta_sh[ng:] == [0, 1, 0, 1])
