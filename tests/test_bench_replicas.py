"""The replica path of bench.py on CPU: two gloo ranks, each with its own
step time; the job time is the slowest rank's and the throughput counts the
units of every rank.  No GPU."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    r, w = bench.init_dist("gloo")
    assert (r, w) == (rank, world)
    local_ms = 10.0 + 5.0 * rank          # rank 1 is slower
    ms = bench.max_over_ranks(local_ms)
    bench.barrier()
    out[rank] = (ms, bench.aggregate(2.0, ms / 1e3, w))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_replicas_take_the_max_and_sum_units():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    assert out[0][0] == out[1][0] == 15.0
    assert out[0][1] == pytest.approx(2.0 * world / 0.015)


def test_single_process_aggregate():
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.aggregate(1.0, 0.5, 1) == 2.0
