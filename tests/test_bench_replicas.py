"""The multi-GPU path of the bench is replicas only: each rank times its own
copy of the step and rank 0 reports all replicas' work over the slowest
rank's time. Its host logic runs here as two gloo ranks on the CPU."""

import os
import socket
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port),
                       "RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench.dist_info()
        # rank 0 is slower at prefill, rank 1 at decode; only rank 1 ran a copy phase
        phases = {"prefill": 1.0 + (rank == 0), "decode": 0.5 + 0.25 * (rank == 1)}
        if rank == 1:
            phases["copy"] = 0.1
        got, step = bench.max_over_ranks(phases, sum(phases.values()), "cpu")
        out[rank] = (w, r, local, got, step)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_to_the_slowest():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        w, r, local, got, step = res[rank]
        assert (w, r, local) == (world, rank, rank)
        assert got["prefill"] == pytest.approx(2.0) and got["decode"] == pytest.approx(0.75)
        assert step == pytest.approx(max(2.0 + 0.5, 1.0 + 0.75 + 0.1))
    # a phase only rank 1 ran reaches rank 1 (rank 0 never asked for it)
    assert res[1][3]["copy"] == pytest.approx(0.1) and "copy" not in res[0][3]


def test_whole_job_rate_counts_every_replica():
    sys.path.insert(0, ROOT)
    import bench

    # four replicas each moving 1 GB, the slowest taking 2 ms: 2 TB/s for the job
    assert bench.whole_job_rate(1e9, 4, 2.0) == pytest.approx(2e12)
    assert bench.max_over_ranks({"decode": 1.5}, 1.5, "cpu") == ({"decode": 1.5}, 1.5)
