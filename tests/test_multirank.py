"""Host-side logic of the multi-rank benchmark run (CPU, gloo, world size 2).

Each rank runs an independent replica of the block; ranks meet only to agree on
the slowest rank's time, and only rank 0 prints.  These tests exercise that
logic with two gloo processes on 127.0.0.1 -- no GPU, no NCCL.
"""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench.dist_env()
        slowest = bench.max_over_ranks(10.0 + 5.0 * rank)      # rank 1 is the slow one
        value = bench.job_tflops(10299e9, slowest, ws)
        dist.barrier()
        out[rank] = (ws, r, local, slowest, value)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    assert sorted(res) == [0, 1]
    for rank, (ws, r, local, slowest, value) in res.items():
        assert (ws, r, local) == (2, rank, rank)
        assert slowest == 15.0                      # max over ranks
        assert value == pytest.approx(2 * 10299e9 / 15e-3 / 1e12)   # whole-job throughput


def test_single_process_needs_no_process_group():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert not dist.is_initialized()
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_tflops(1e12, 1000.0, 1) == pytest.approx(1.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")

    class Args:
        steps, warmup = 3, 1
    bench.run_reference(Args())        # rank 1: returns at once, prints nothing
    assert capsys.readouterr().out == ""
