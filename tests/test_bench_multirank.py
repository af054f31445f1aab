"""bench.py's multi-process path (independent replicas, one per GPU) on the
CPU with the gloo backend, world size 2: the job time is the slowest rank's
and the rate sums every rank's parameters."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ws, r, local = bench.dist_env()
    assert (ws, r, local) == (world, rank, rank)
    # rank 0 took 100 ms for 1000 params x 10 steps, rank 1 took 250 ms for 3000 params
    ms, value = bench.aggregate([100.0, 250.0][rank], [1000, 3000][rank], 10)
    out[rank] = (ms, value)
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation_gloo():
    port = _free_port()
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(2):
        ms, value = out[r]
        assert ms == 250.0
        assert value == pytest.approx((1000 + 3000) * 10 / 0.25)


def test_single_process_aggregation():
    sys.path.insert(0, ROOT)
    import bench
    ms, value = bench.aggregate(50.0, 2000, 4)
    assert ms == 50.0 and value == pytest.approx(2000 * 4 / 0.05)
