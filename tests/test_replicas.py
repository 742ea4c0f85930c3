"""The N > 1 path of bench.py on CPU: independent replicas, no data-path collective, the job's
time is the slowest rank's and its rate counts every replica's rows (world_size 2, gloo)."""

import os
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local = 2.0 + rank  # rank 1 is the slower replica
        job = bench.max_over_ranks(local, dist, "cpu")
        rate = bench.whole_job_rate(world, 33720, 3, job)
        dist.barrier()
        out[rank] = (job, rate)
    finally:
        dist.destroy_process_group()


def test_two_replicas_report_slowest_time_and_all_rows():
    port = 29500 + os.getpid() % 1000
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(2, port, out), nprocs=2, join=True)
        res = dict(out)
    for r in (0, 1):
        job, rate = res[r]
        assert job == 3.0  # max over ranks
        assert rate == pytest.approx(2 * 33720 * 3 / 3.0)


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(1.25) == 1.25
    assert bench.whole_job_rate(1, 1000, 2, 0.5) == 4000.0
