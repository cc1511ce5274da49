"""The multi-GPU path of the benchmark is replicas only: each rank runs a full
product and the job's throughput uses the slowest rank's time.  This checks the
cross-rank aggregation with two gloo ranks on the CPU (no GPU, no collective
on any data path)."""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        t = bench.max_over_ranks(times[rank], world, "cpu")
        out[rank] = (t, bench.job_tflops(2.0 * 8192 ** 3, 10, world, t))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_two_ranks():
    world = 2
    times = [120.0, 150.0]
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank, args=(world, _free_port(), times, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 150.0
    want = 2.0 * 8192 ** 3 * 10 * 2 / 0.150 / 1e12
    assert res[0][1] == pytest.approx(want)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5
    assert bench.job_tflops(2e12, 1, 1, 1000.0) == pytest.approx(2.0)
