"""The multi-process host logic of bench.py on CPU (gloo, world size 2):
each rank runs its own replica of the workload (the path shards by query
rows / sequences with no exchange), the slowest rank's time is the step time
(max over ranks), and the throughput counts the units of every rank."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    w, r, _ = bench.dist_setup(None)
    assert (w, r) == (world, rank)
    bench.barrier(w)
    ms = 10.0 + 5.0 * rank          # rank 1 is the slow one
    slowest = bench.max_over_ranks(ms, w)
    tokens_per_rank = 4096
    value = tokens_per_rank * w / (slowest / 1e3)
    q.put((rank, slowest, value))
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_rank_timing_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(100)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=5) for _ in range(2))
    for rank, slowest, value in res:
        assert slowest == 15.0
        assert abs(value - 2 * 4096 / 0.015) < 1e-6
