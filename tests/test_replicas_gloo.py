"""The multi-rank path of bench.py (replicas only: each rank runs the whole workload on its own
GPU, the job time is the slowest rank's) with two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_ms = [3.0, 5.0][rank]
    bench.barrier(world)
    ms = bench.max_over_ranks(local_ms, world, device="cpu")
    value = bench.job_us_per_matrix(ms, launches_per_rank=100, world=world)
    q.put((rank, ms, value))
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, value in out:
        assert ms == 5.0                      # max over ranks
        assert value == pytest.approx(5.0 * 1e3 / 200)  # 200 matrices job-wide


def test_single_rank_value():
    import bench
    assert bench.max_over_ranks(7.0, 1) == 7.0
    assert bench.job_us_per_matrix(2.0, 10, 1) == pytest.approx(200.0)
