"""The benchmark's multi-rank aggregation on CPU: two gloo ranks, each timing
its own (weak-scaled) share; the whole-job value is the tokens of all ranks
over the slowest rank's time."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    assert bench.dist_env() == (world, rank, rank)
    bench.barrier(torch.device("cpu"))
    elapsed = [2.0, 3.0][rank]
    value, tmax = bench.aggregate(1000, elapsed, world, torch.device("cpu"))
    q.put((rank, value, tmax))
    dist.destroy_process_group()


def test_two_rank_aggregation_takes_max_time_and_total_tokens():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    for rank, value, tmax in res:
        assert tmax == pytest.approx(3.0)
        assert value == pytest.approx(2 * 1000 / 3.0)
