"""Host-side logic of the multi-rank benchmark run (CPU, gloo, world size 2).

Each rank runs an independent replica of the block; ranks meet only to agree on
the slowest rank's time, and only rank 0 prints.  These tests exercise that
logic with two gloo processes on 127.0.0.1 -- no GPU, no NCCL.  One more checks,
with the oracle, the data-parallel reading of the block (token rows split across
ranks need one exchange, the sum of the weight gradients), and one the
tensor-parallel reading (hidden columns split across ranks: y and dx are sums of
partial products).  The managers are started with spawn: the oracle's OpenMP
threads make a later fork unsafe.
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
    with mp.get_context("spawn").Manager() as m:
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


def _dp_worker(rank, world, port, out):
    """Rank `rank` takes its share of the token rows through the oracle's block."""
    import sys
    sys.path.insert(0, ROOT)
    import torch
    import oracle
    from bwd_gemm_epilogue_gb300 import workloads
    from bwd_gemm_epilogue_gb300.workloads import Shape
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        s, x, W1, W2, dy = workloads.make_block(Shape(96, 64, 80, 48), seed=7)
        rows = slice(rank * s.M // world, (rank + 1) * s.M // world)
        xs, dys = x[rows].contiguous(), dy[rows].contiguous()
        preact, _, y = oracle.fwd(xs, W1, W2)
        # the saved preact is bf16-rounded: back to bf16 exactly, like the other inputs
        _, _, _, dx, dW1, dW2 = oracle.bwd_full(xs, W1, W2, torch.from_numpy(preact).to(torch.bfloat16), dys)
        dW1, dW2 = torch.from_numpy(dW1), torch.from_numpy(dW2)
        dist.all_reduce(dW1)                     # the one exchange the row split needs
        dist.all_reduce(dW2)
        ys = [torch.empty_like(torch.from_numpy(y)) for _ in range(world)]
        dxs = [torch.empty_like(torch.from_numpy(dx)) for _ in range(world)]
        dist.all_gather(ys, torch.from_numpy(y))
        dist.all_gather(dxs, torch.from_numpy(dx))
        out[rank] = (torch.cat(ys).numpy(), torch.cat(dxs).numpy(), dW1.numpy(), dW2.numpy())
    finally:
        dist.destroy_process_group()


def test_row_shards_with_summed_weight_gradients_give_the_full_batch():
    # Data parallelism over token rows: y and dx are row-wise, so each rank's rows are
    # final; dW1 and dW2 are sums over rows, so the ranks' partial sums add up to the
    # full batch's (up to the fp64 order of the additions).
    import sys
    sys.path.insert(0, ROOT)
    import numpy as np
    import torch
    import oracle
    from bwd_gemm_epilogue_gb300 import workloads
    from bwd_gemm_epilogue_gb300.workloads import Shape
    oracle.build()                               # once, before the ranks load it
    world = 2
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_dp_worker, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    _, x, W1, W2, dy = workloads.make_block(Shape(96, 64, 80, 48), seed=7)
    preact, _, y = oracle.fwd(x, W1, W2)
    preact = torch.from_numpy(preact).to(torch.bfloat16)
    _, _, _, dx, dW1, dW2 = oracle.bwd_full(x, W1, W2, preact, dy)
    for rank in range(world):
        ys, dxs, dW1s, dW2s = res[rank]
        np.testing.assert_array_equal(ys, y)
        np.testing.assert_array_equal(dxs, dx)
        np.testing.assert_allclose(dW1s, dW1, rtol=1e-12, atol=1e-12 * np.abs(dW1).max())
        np.testing.assert_allclose(dW2s, dW2, rtol=1e-12, atol=1e-12 * np.abs(dW2).max())
    # a rank that skipped the exchange would hold only its own rows' share
    _, _, _, _, dW1_half, _ = oracle.bwd_full(x[:48].contiguous(), W1, W2, preact[:48].contiguous(),
                                               dy[:48].contiguous())
    assert np.abs(dW1_half - dW1).max() > 1e-3 * np.abs(dW1).max()


class _OracleShardCompute:
    """The shard products on the host (the oracle), for the tensor-parallel module's CPU path."""

    def __init__(self, rows_per_chunk):
        self.rows = rows_per_chunk

    def chunk_rows(self, M, n_chunks):
        return self.rows

    def fwd(self, x, W1s, W2s, n_chunks, events):
        import torch
        import oracle
        preact, _, y = oracle.fwd(x, W1s, W2s)
        return torch.from_numpy(preact).to(torch.bfloat16), torch.from_numpy(y)

    def bwd(self, x, W1s, W2s, preact, dy, event):
        import torch
        import oracle
        _, _, _, dx, dW1s, dW2s = oracle.bwd_full(x, W1s, W2s, preact, dy)
        return torch.from_numpy(dx), torch.from_numpy(dW1s), torch.from_numpy(dW2s)


def _tp_worker(rank, world, port, out, reduce):
    """Rank `rank` holds hidden columns J_r: W1 rows J_r (left) and H + J_r (gate), W2 columns J_r;
    the library's tensor-parallel module chunks and reduces its partial y and dx."""
    import sys
    sys.path.insert(0, ROOT)
    import torch
    from bwd_gemm_epilogue_gb300 import workloads
    from bwd_gemm_epilogue_gb300.tensor_parallel import TensorParallelSwiGLU, shard_bounds
    from bwd_gemm_epilogue_gb300.workloads import Shape
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        s, x, W1, W2, dy = workloads.make_block(Shape(64, 48, 96, 40), seed=11)
        j0, Hs = shard_bounds(s.H, world, rank)
        J = slice(j0, j0 + Hs)
        W1r = torch.cat([W1[J], W1[s.H:][J]]).contiguous()
        W2r = W2[:, J].contiguous()
        tp = TensorParallelSwiGLU(W1r, W2r, n_chunks=3, reduce=reduce, compute=_OracleShardCompute(24))
        y, preact = tp.forward(x)                     # chunked reduction after the down projection
        dx, dW1r, dW2r = tp.backward(x, preact, dy)   # chunked reduction of dx
        out[rank] = (y.numpy(), dx.numpy(), dW1r.numpy(), dW2r.numpy(), [tp.owner(c) for c in range(3)])
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("reduce", ["all_reduce", "reduce_scatter"])
def test_hidden_column_shards_with_summed_outputs_give_the_full_block(reduce):
    # Tensor parallelism over the hidden dimension: each rank's left/gate columns are a
    # complete SwiGLU of their own, so y and dx are sums of per-rank partial products and
    # each rank's weight gradients are its slices of the full ones.  The reductions go
    # through the library's tensor-parallel module in three row chunks of 24, 24 and 16 rows.
    import sys
    sys.path.insert(0, ROOT)
    import numpy as np
    import torch
    import oracle
    from bwd_gemm_epilogue_gb300 import workloads
    from bwd_gemm_epilogue_gb300.workloads import Shape
    oracle.build()
    world = 2
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_tp_worker, args=(world, _free_port(), out, reduce), nprocs=world, join=True)
        res = dict(out)
    s, x, W1, W2, dy = workloads.make_block(Shape(64, 48, 96, 40), seed=11)
    preact, _, y = oracle.fwd(x, W1, W2)
    _, _, _, dx, dW1, dW2 = oracle.bwd_full(x, W1, W2, torch.from_numpy(preact).to(torch.bfloat16), dy)
    half = s.H // world
    chunks = [slice(0, 24), slice(24, 48), slice(48, 64)]
    for rank in range(world):
        ys, dxs, dW1r, dW2r, owners = res[rank]
        assert owners == [0, 1, 0]
        for c, rows in enumerate(chunks):
            if reduce == "reduce_scatter" and owners[c] != rank:
                continue                               # another rank receives this chunk's sum
            np.testing.assert_allclose(ys[rows], y[rows], rtol=1e-12, atol=1e-12 * np.abs(y).max())
            np.testing.assert_allclose(dxs[rows], dx[rows], rtol=1e-12, atol=1e-12 * np.abs(dx).max())
        J = slice(rank * half, (rank + 1) * half)
        np.testing.assert_allclose(dW1r[:half], dW1[J], rtol=1e-12, atol=1e-12 * np.abs(dW1).max())
        np.testing.assert_allclose(dW1r[half:], dW1[s.H:][J], rtol=1e-12, atol=1e-12 * np.abs(dW1).max())
        np.testing.assert_allclose(dW2r, dW2[:, J], rtol=1e-12, atol=1e-12 * np.abs(dW2).max())
    if reduce == "reduce_scatter":                      # a chunk another rank owns holds a partial sum only
        assert np.abs(res[1][0][chunks[0]] - y[chunks[0]]).max() > 1e-3 * np.abs(y).max()


def test_pairing_left_and_gate_of_different_ranks_is_not_the_block():
    import sys
    sys.path.insert(0, ROOT)
    import numpy as np
    import torch
    import oracle
    from bwd_gemm_epilogue_gb300 import workloads
    from bwd_gemm_epilogue_gb300.workloads import Shape
    s, x, W1, W2, dy = workloads.make_block(Shape(64, 48, 96, 40), seed=11)
    half = s.H // 2
    # pairing a rank's left columns with another rank's gate columns is not the block
    W1_wrong = torch.cat([W1[:half], W1[s.H + half:]]).contiguous()
    _, _, y_wrong = oracle.fwd(x, W1_wrong, W2[:, :half].contiguous())
    _, _, y_right = oracle.fwd(x, torch.cat([W1[:half], W1[s.H:s.H + half]]).contiguous(), W2[:, :half].contiguous())
    assert np.abs(y_wrong - y_right).max() > 1e-2 * np.abs(y_right).max()
