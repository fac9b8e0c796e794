"""Replicas on N>1 GPUs: bench.py's host logic (max-over-ranks time and
whole-job throughput) checked with two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    ws, r, local = bench.dist_env()
    assert (ws, r, local) == (world, rank, rank)
    ms_rank = [2.0, 5.0][rank]
    value, ms = bench.aggregate(64, ms_rank, world)
    bench.barrier()
    q.put((rank, value, ms))
    dist.destroy_process_group()


def test_two_rank_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, value, ms in res:
        assert ms == 5.0                       # the slowest rank's time
        assert value == pytest.approx(64 * 2 / 5e-3)  # all ranks' tokens over it


def test_single_process_aggregation():
    import bench

    assert not dist.is_initialized()
    value, ms = bench.aggregate(10, 4.0, 1)
    assert ms == 4.0 and value == pytest.approx(2500.0)
