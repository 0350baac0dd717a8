"""The multi-GPU path is replicas only; its host logic (max-over-ranks step time,
whole-job throughput) runs on CPU ranks over gloo, world size 2."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms, tps = bench.aggregate(10.0 + 5.0 * rank, 64, world)
    out[rank] = (ms, tps)
    dist.destroy_process_group()


def test_aggregate_two_ranks():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    out = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(2):
        ms, tps = out[r]
        assert ms == 15.0                       # slowest rank
        assert abs(tps - 2 * 64 / 0.015) < 1e-6  # every rank's tokens


def test_aggregate_single():
    import bench
    assert bench.aggregate(2.0, 4, 1) == (2.0, 2000.0)
