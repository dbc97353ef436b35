"""Host logic of the N > 1 benchmark path (replicas, weak scaling) on CPU:
two gloo ranks, the slowest rank's time is what every rank reports."""
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


def _rank(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        ms = bench.max_over_ranks(times[rank], world, torch.device("cpu"))
        out[rank] = (ms, bench.whole_job_tflops(1e12, world, ms))
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_weak_scaling_value():
    world = 2
    times = [3.0, 5.0]
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank, args=(world, _free_port(), times, out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        ms, tflops = res[r]
        assert ms == 5.0                                  # slowest rank
        assert tflops == pytest.approx(2 * 1e12 / 5e-3 / 1e12)


def test_single_rank_passthrough():
    import bench
    assert bench.max_over_ranks(1.25, 1, torch.device("cpu")) == 1.25
    assert bench.whole_job_tflops(2e12, 1, 1.0) == pytest.approx(2000.0)


def test_rotating_sets_exceed_l2():
    # every workload rotates through input sets that together hold >= 2 x L2
    import bench
    for name in bench.WORKLOADS:
        n = bench.n_rotating_sets(name)
        assert n >= 2
        assert n * bench.step_bytes(name) >= 2 * bench.L2_BYTES or n == 4096
