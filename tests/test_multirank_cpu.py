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


def _replica_worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import time

    import bench

    def run():                                # a CPU stand-in for one replica's timed steps
        t0 = time.perf_counter()
        time.sleep(0.05 * (rank + 1))         # rank 1 is the slow replica
        return (time.perf_counter() - t0) * 1e3
    local_ms, slowest_ms = bench.replica_timing(run, world, lambda: None, dist.barrier)
    out[rank] = (local_ms, slowest_ms, bench.job_value(2.0e12, slowest_ms, world))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_replicas_run_the_timed_region_end_to_end():
    """Each rank runs its own replica between barriers; every rank reports
    the slowest rank's time, and the job value counts both replicas' work."""
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_replica_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] < res[1][0]                      # rank 0 ran faster
    assert res[0][1] == res[1][1] == res[1][0]        # both report rank 1's time
    assert abs(res[0][2] - 2 * 2.0e12 / res[1][0] / 1e9) < 1e-6


def test_more_gpus_than_visible_is_refused():
    """--gpus N outside torchrun relaunches one replica per GPU, and refuses
    (exit code 2) when fewer GPUs are visible -- never a silent 1-GPU run."""
    import subprocess
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    env.pop("WORLD_SIZE", None)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 2 and "asks for 2 GPUs" in r.stderr


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert abs(bench.job_value(2.0e12, 4.0, 1) - 500.0) < 1e-9
