"""The N-GPU benchmark path on CPU: two gloo ranks agree on the slowest rank's
step time and on the whole-job throughput (replicas, weak scaling)."""
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


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    t = bench.max_over_ranks(0.010 + 0.005 * rank, "cpu")
    out[rank] = (t, bench.job_throughput(world, 1000, t))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_step():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank, args=(world, _free_port(), out), nprocs=world, start_method="spawn", join=True)
    assert sorted(out.keys()) == [0, 1]
    for r in range(world):
        t, v = out[r]
        assert t == pytest.approx(0.015)
        assert v == pytest.approx(2 * 1000 / 0.015)


def test_single_process_is_its_own_maximum():
    import bench
    assert bench.max_over_ranks(0.25, "cpu") == 0.25
