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


def test_layer_count_exceeds_l2_three_times_over():
    """Back-to-back timing: between two reads of one layer, the other layers' rows
    fill L2 at least three times; tiny steps or caches that do not fit fall back to
    isolated steps (0)."""
    l2, free = 136_000_000, 280 << 30    # the GB300 reports a 136 MB L2
    step_c3, cache_c3 = 38_300_000, 1_224_736_768
    nl = bench.plan_layers(step_c3, cache_c3, l2, free)
    assert nl == 12
    assert (nl - 1) * step_c3 >= bench.L2_TURNOVER * l2
    assert (nl - 2) * step_c3 < bench.L2_TURNOVER * l2      # the smallest such count
    assert bench.plan_layers(75_000, 10_000_000, l2, free) == 0          # batch-1 step
    assert bench.plan_layers(step_c3, cache_c3, l2, 8 << 30) == 0        # no room
    assert bench.plan_layers(500 << 20, 1 << 30, l2, free) == 2          # step > 3 x L2
