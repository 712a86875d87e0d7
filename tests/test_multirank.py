"""The N > 1 path of the benchmark on CPU: two ranks over gloo (127.0.0.1) agree on the
slowest rank's time and report the whole job's throughput (replicas only: every rank runs its
own copy of the step, no data is exchanged)."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def worker(rank, world, port, out):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [120.0, 180.0][rank]          # rank 1 is the slow one
    slowest = bench.max_over_ranks(local_ms, dist, torch.device("cpu"))
    gbs, ips = bench.job_throughput(1_000_000_000, 64, world, slowest, steps=10)
    out[rank] = (slowest, gbs, ips)
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_gloo():
    import torch.multiprocessing as mp
    world = 2
    port = free_port()
    manager = mp.Manager()
    out = manager.dict()
    mp.spawn(worker, args=(world, port, out), nprocs=world, join=True)
    assert out[0] == out[1]
    slowest, gbs, ips = out[0]
    assert slowest == 180.0
    # 10 steps in 180 ms -> 18 ms a step; 2 ranks x 1 GB each per step
    assert abs(gbs - 2 * 1.0 / 0.018) < 1e-9
    assert abs(ips - 2 * 64 / 0.018) < 1e-6


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(42.0, None, None) == 42.0
    gbs, ips = bench.job_throughput(2_000_000_000, 8, 1, 1000.0, steps=100)
    assert abs(gbs - 200.0) < 1e-9 and abs(ips - 800.0) < 1e-9
