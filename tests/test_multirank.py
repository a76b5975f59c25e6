"""The multi-rank host logic of bench.py on CPU (gloo, world size 2): each
rank runs its own replica, and the job time is the slowest rank's."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        assert (r, w, local) == (rank, world, rank)
        # rank 1 is the slow one: every rank must see its time
        t = bench.max_over_ranks(10.0 + 5.0 * rank, world)
        results[rank] = t
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    port = _free_port()
    with mp.Manager() as m:
        results = m.dict()
        mp.spawn(_worker, args=(2, port, results), nprocs=2, join=True)
        assert dict(results) == {0: 15.0, 1: 15.0}


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import bench
    import workloads
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class Args:
        steps, warmup = 3, 3
    bench.run_reference(Args, workloads.WORKLOADS[1])
    assert capsys.readouterr().out == ""
