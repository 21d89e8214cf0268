"""Host logic of multi-GPU benchmarking, run as two gloo ranks on the CPU.

Each rank runs an independent replica of the workload (weak scaling, no
collective on the data path); the reported throughput is the total work of
all ranks over the slowest rank's time.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t_max, flops = bench.aggregate(1.0 + rank, 10.0 * (rank + 1))
        out[rank] = (t_max, flops)
        assert bench.dist_env()[:2] == (world, rank)
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregate():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
        assert all(p.exitcode == 0 for p in procs)
        for r in range(2):
            assert out[r] == (2.0, 30.0)   # slowest rank's time, all ranks' work


def test_single_process_aggregate_is_identity():
    import bench
    assert bench.aggregate(0.5, 7.0) == (0.5, 7.0)
