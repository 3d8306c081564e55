"""The multi-GPU path is independent replicas (no data-path collective):
the bench takes the slowest rank's time and reports the whole job's rate.
Checked here with two gloo ranks on CPU."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # Rank r "measured" (1 + r) ms for the kernel and (5 - r) ms e2e.
        got = bench.max_over_ranks([1.0 + rank, 5.0 - rank])
        out[rank] = got
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_rank, args=(world, port, out), nprocs=world,
                           start_method="spawn", join=True)
        res = dict(out)
    assert res[0] == res[1] == [2.0, 5.0]


def test_single_rank_is_identity():
    assert bench.max_over_ranks([3.5, 1.25]) == [3.5, 1.25]


@pytest.mark.parametrize("world", [1, 2, 8])
def test_whole_job_rate_counts_every_replica(world):
    # Each replica does 2e12 units in 4 ms: 5e14 units/s per replica.
    assert bench.whole_job_rate(2e12, 4.0, world) == pytest.approx(5e14 * world)
