"""The multi-GPU benchmark path on CPU: two gloo ranks.

bench.py runs one replica of the workload per rank (the scan shards over
(b, d) with no exchange, so no data-path collective exists); the only
collectives are the barrier around the timed region and the max over ranks of
the measured time. This checks that aggregation with world_size 2 on gloo.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys
    import torch.distributed as dist
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        local_ms = 10.0 * (rank + 1)                  # rank 1 is the slowest
        slowest = bench.max_over_ranks(local_ms)
        value = bench.job_throughput(1000, 5, world, slowest)
        dist.barrier()
        q.put((rank, slowest, value))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank_and_sum_the_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, slowest, value in got:
        assert slowest == 20.0
        assert value == pytest.approx(2 * 1000 * 5 / 0.020)


def test_single_process_aggregation_is_identity():
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_throughput(100, 2, 1, 4.0) == pytest.approx(100 * 2 / 0.004)
