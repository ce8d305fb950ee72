"""The multi-GPU bench path on CPU: two gloo ranks aggregate their step times with
a max and report whole-job throughput (every rank decodes its own batch; no data
exchange is part of the decode)."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    mine = [1.0 + rank, 10.0 - rank, 3.5]
    got = bench.aggregate_over_ranks(mine, torch.device("cpu"), world)
    q.put((rank, got, bench.job_throughput(world, 32, got[0])))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_aggregation_takes_the_max():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict()
    for _ in range(2):
        rank, got, value = q.get(timeout=120)
        res[rank] = (got, value)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank in (0, 1):
        got, value = res[rank]
        assert got == [2.0, 10.0, 3.5]
        assert abs(value - 2 * 32 / 2e-3) < 1e-6


def test_single_rank_is_identity():
    assert bench.aggregate_over_ranks([4.0, 5.0], torch.device("cpu"), 1) == [4.0, 5.0]
    assert bench.job_throughput(1, 32, 0.01) == 32 / 1e-5
