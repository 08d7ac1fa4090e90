"""The multi-rank timing aggregation of bench.py, on CPU with gloo (world
size 2): the max over ranks and the whole-job throughput."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, _ = bench.dist_env()
        assert (ws, r) == (world, rank)
        seconds = 1.0 + rank              # rank 1 is the slower one
        slowest = bench.max_over_ranks(seconds, ws)
        bench.barrier(ws)
        out[rank] = (slowest, bench.aggregate_throughput(10.0, ws, slowest))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_aggregate_gloo():
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
    # both ranks see the slowest time; throughput = units of all ranks / slowest time
    assert out[0] == out[1] == (2.0, 10.0 * 2 / 2.0)


def test_single_rank_helpers():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.aggregate_throughput(8.0, 1, 2.0) == 4.0
