"""The multi-process path of bench.py on the CPU: world size 2 over gloo (127.0.0.1).

On a GPU node the benchmark runs one independent replica per GPU (the path has no exchange step),
times each rank, takes the maximum over ranks and reports the units of all ranks over that time.
This test runs the same aggregation with two gloo ranks on the host.
"""
import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, queue):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    seconds = [0.030, 0.050][rank]  # rank 1 is the slower replica
    slowest = bench.max_over_ranks(seconds, world)
    queue.put((rank, slowest, bench.job_throughput(1024, slowest, world)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_max_over_ranks_and_job_throughput():
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    results = [queue.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, tput in results:
        assert slowest == pytest.approx(0.050)
        assert tput == pytest.approx(2 * 1024 / 0.050)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(0.25, 1) == 0.25
    assert bench.job_throughput(10, 2.0, 1) == 5.0
