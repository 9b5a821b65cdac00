"""The N > 1 bench path on CPU: world-size-2 gloo process groups.

Every rank runs an independent replica; the reported time is the slowest
rank's (max over ranks) and the whole-job rate counts every rank's units.
The reference arm runs on rank 0 only."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, values, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        m = bench.max_over_ranks(values[rank])
        dist.barrier()
        out[rank] = m
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_processes():
    world, port = 2, _free_port()
    values = [3.25, 7.5]
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, port, values, out), nprocs=world, join=True)
        assert out[0] == out[1] == max(values)


def test_max_over_ranks_single_process_is_identity():
    assert bench.max_over_ranks(4.0) == 4.0


def test_whole_job_rate_counts_every_rank():
    # 2 ranks x 10 steps x 1e6 units in 20 ms (the slowest rank) = 1e9 units/s
    assert bench.whole_job_rate(1e6, 2, 10, 20.0) == pytest.approx(1e9)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    assert bench.run_reference(None) is None     # no work, no line on rank 1
