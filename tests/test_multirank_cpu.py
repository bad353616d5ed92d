"""The N > 1 path of bench.py (independent replicas, one per rank) on CPU with
two gloo ranks: the step time is the slowest rank's and the job value sums
every replica's work."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    local_ms = 10.0 + 5.0 * rank              # rank 1 is the slow replica
    ms = bench.max_over_ranks(local_ms, world)
    out[rank] = (ms, bench.job_value(1.0e12, ms, world))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank_and_sum_the_work():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 15.0
    # 2 replicas x 1 TFLOP each in 15 ms
    assert abs(res[0][1] - 2.0e12 / 15.0 / 1e9) < 1e-9
    assert res[0] == res[1]


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert abs(bench.job_value(2.0e12, 4.0, 1) - 500.0) < 1e-9
