"""Tensor-parallel shards of the block through the C ABI, against the fp64 oracle.

Rank r of `world` owns hidden units J = [j0, j0 + Hs): W1 rows J and H + J, W2 columns J
("Lesson 24: MLP, GEMM and operator fusion in the Transformer", section 33).  On one GPU
every rank's shard runs in turn; their partial y and dx must add up to the block's, and
their weight gradients, written back into full-size tensors, must be the block's.  The
oracle computes the full block from the same inputs (its preact feeds every shard's
backward); nothing it reads comes from the GPU.
"""
import os
import socket

import numpy as np
import pytest
import torch

import oracle
from bwd_gemm_epilogue_gb300 import workloads
from bwd_gemm_epilogue_gb300.tensor_parallel import shard_bounds
from bwd_gemm_epilogue_gb300.workloads import Shape
from helpers import ensure_library, parity

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def b():
    ensure_library()
    from bwd_gemm_epilogue_gb300 import binding
    binding.lib()
    return binding


def dev(t):
    return t.cuda().contiguous()


def shard_cols(H, j0, Hs):
    """Columns of preact / grad_preact that belong to the shard: left J, then gate H + J."""
    return np.concatenate([np.arange(j0, j0 + Hs), H + np.arange(j0, j0 + Hs)])


def run_shards(b, s, world, x, W1, W2, dy, pre_in, n_chunks=3):
    """Every rank's shard forward and backward on this GPU; returns per-rank outputs."""
    xd, W1d, W2d, dyd = dev(x), dev(W1), dev(W2), dev(dy)
    out = []
    for r in range(world):
        j0, Hs = shard_bounds(s.H, world, r)
        W1s, W2s = b.swiglu_mlp_tp_shard_pack(W1d, W2d, j0, Hs)
        # the pack is the row / column selection of the lesson's column-parallel split
        assert torch.equal(W1s, torch.cat([W1d[j0:j0 + Hs], W1d[s.H + j0:s.H + j0 + Hs]]))
        assert torch.equal(W2s, W2d[:, j0:j0 + Hs])
        events = [torch.cuda.Event() for _ in range(n_chunks)]
        pre_s, y_p = b.swiglu_mlp_tp_fwd(xd, W1s, W2s, n_chunks=n_chunks, chunk_events=events)
        ev = torch.cuda.Event()
        pin = dev(pre_in[:, torch.from_numpy(shard_cols(s.H, j0, Hs))])
        dx_p, dW1s, dW2s = b.swiglu_mlp_tp_bwd(xd, W1s, W2s, pin, dyd, dx_event=ev)
        torch.cuda.synchronize()
        assert all(e.query() for e in events) and ev.query()
        out.append(dict(j0=j0, Hs=Hs, pre=pre_s, y=y_p, dx=dx_p, dW1=dW1s, dW2=dW2s, W1s=W1s, W2s=W2s))
    assert b.swiglu_mlp_device_status() == 0
    return out


CASES = [(2, Shape(300, 256, 512, 264)), (4, Shape(640, 128, 1024, 256)), (2, Shape(40, 128, 512, 256)),
         (2, Shape(129, 64, 272, 96))]


@pytest.mark.parametrize("world,s", CASES, ids=lambda v: str(v) if isinstance(v, int) else f"M{v.M}_D{v.D}_H{v.H}_Do{v.Dout}")
def test_shards_add_up_to_the_block(b, world, s):
    _, x, W1, W2, dy = workloads.make_block(s, seed=90 + world + s.M)
    p_ref, _, y_ref = oracle.fwd(x, W1, W2)
    pre = torch.from_numpy(p_ref).to(torch.bfloat16)
    _, _, _, dx_ref, dW1_ref, dW2_ref = oracle.bwd_full(x, W1, W2, pre, dy)
    shards = run_shards(b, s, world, x, W1, W2, dy, pre)
    y = sum(o["y"].float() for o in shards)
    dx = sum(o["dx"].float() for o in shards)
    dW1 = torch.full_like(W1, float("nan")).cuda()
    dW2 = torch.full_like(W2, float("nan")).cuda()
    for o in shards:
        cols = shard_cols(s.H, o["j0"], o["Hs"])
        parity(o["pre"], p_ref[:, cols], f"preact of shard j0={o['j0']}")
        b.swiglu_mlp_tp_shard_unpack_grads(o["dW1"], o["dW2"], dW1, dW2, o["j0"])
    torch.cuda.synchronize()
    parity(y, y_ref, "sum of the partial y")
    parity(dx, dx_ref, "sum of the partial dx")
    parity(dW1, dW1_ref, "dW1 from the shards")      # every row written (no NaN left)
    parity(dW2, dW2_ref, "dW2 from the shards")


def test_chunks_and_dx_event_change_no_bits(b):
    # The chunked down projection and the separate dx launch compute every tile as the
    # one-piece forward / grouped backward do: the same bits.
    s = Shape(1000, 256, 768, 320)
    _, x, W1, W2, dy = workloads.make_block(s, seed=97)
    xd, W1d, W2d, dyd = dev(x), dev(W1), dev(W2), dev(dy)
    j0, Hs = shard_bounds(s.H, 3, 1)
    W1s, W2s = b.swiglu_mlp_tp_shard_pack(W1d, W2d, j0, Hs)
    pre1, y1 = b.swiglu_mlp_tp_fwd(xd, W1s, W2s, n_chunks=1)
    ev = [torch.cuda.Event() for _ in range(5)]
    pre5, y5 = b.swiglu_mlp_tp_fwd(xd, W1s, W2s, n_chunks=5, chunk_events=ev)
    pre_b, y_b = b.swiglu_mlp_fwd(xd, W1s, W2s)
    dxa, dW1a, dW2a = b.swiglu_mlp_tp_bwd(xd, W1s, W2s, pre1, dyd)
    dxb, dW1b, dW2b = b.swiglu_mlp_tp_bwd(xd, W1s, W2s, pre1, dyd, dx_event=torch.cuda.Event())
    torch.cuda.synchronize()
    assert b.swiglu_mlp_device_status() == 0
    assert b.swiglu_mlp_tp_chunk_rows(s.M, 5) == 256          # whole 256-row tiles; the last chunk is empty
    for a, c in ((pre1, pre5), (y1, y5), (y1, y_b), (pre1, pre_b), (dxa, dxb), (dW1a, dW1b), (dW2a, dW2b)):
        assert torch.equal(a, c)


def test_shard_arguments_are_checked(b):
    W1 = torch.zeros(2 * 64, 32, dtype=torch.bfloat16, device="cuda")
    W2 = torch.zeros(16, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(RuntimeError, match="j0 \\+ Hs <= H"):
        b.swiglu_mlp_tp_shard_pack(W1, W2, 40, 32)            # past the last hidden unit
    with pytest.raises(RuntimeError, match="UNSUPPORTED_SHAPE"):
        b.swiglu_mlp_tp_shard_pack(W1, W2, 4, 16)             # j0 not a multiple of 8
    x = torch.zeros(300, 32, dtype=torch.bfloat16, device="cuda")
    W1s, W2s = b.swiglu_mlp_tp_shard_pack(W1, W2, 0, 32)
    with pytest.raises(RuntimeError, match="n_chunks"):
        b.swiglu_mlp_tp_fwd(x, W1s, W2s, n_chunks=0)


def test_target_shape_two_shards_every_tile(b):
    # The pages' target block split over two ranks (Hs = 7168): rows of every 256-row tile
    # and hidden units of every 256-column tile of each shard, sampled.
    from test_gpu_parity import tile_indices
    s, x, W1, W2, dy = workloads.make_block("target")
    pre = workloads.make_preact(s, workloads.CONFIGS["target"]["seed"])
    shards = run_shards(b, s, 2, x, W1, W2, dy, pre, n_chunks=4)
    rows = tile_indices(s.M, 5)
    _, _, y_ref = oracle.fwd(x, W1, W2, rows=rows)
    _, _, _, dx_ref = oracle.bwd_rows(W1, W2, pre, dy, rows=rows)
    parity(sum(o["y"][rows].float() for o in shards), y_ref, "target y[rows], two shards")
    parity(sum(o["dx"][rows].float() for o in shards), dx_ref, "target dx[rows], two shards")
    cols = tile_indices(s.H, 6)
    dW2c_ref, dW1l_ref, dW1g_ref = oracle.bwd_cols(x, W2, pre, dy, cols=cols)
    for o in shards:
        k = np.where((cols >= o["j0"]) & (cols < o["j0"] + o["Hs"]))[0]
        local = torch.from_numpy(cols[k] - o["j0"])
        parity(o["dW2"][:, local].T, dW2c_ref[k], f"dW2 shard j0={o['j0']}")
        parity(o["dW1"][local], dW1l_ref[k], f"dW1 left shard j0={o['j0']}")
        parity(o["dW1"][o["Hs"] + local], dW1g_ref[k], f"dW1 gate shard j0={o['j0']}")


# ---------------------------------------------------------------------------- the reduction on gloo ranks

def _free_port():
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


class _StoredCompute:
    """Returns a rank's shard outputs that the library computed on the GPU (copied to host)."""

    def __init__(self, part, rows):
        self.part, self.rows = part, rows

    def chunk_rows(self, M, n_chunks):
        return self.rows

    def fwd(self, x, W1s, W2s, n_chunks, events):
        return self.part["pre"].clone(), self.part["y"].clone()

    def bwd(self, x, W1s, W2s, preact, dy, event):
        return self.part["dx"].clone(), self.part["dW1"].clone(), self.part["dW2"].clone()


def _gloo_rank(rank, world, port, parts, rows, out):
    import sys
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    from bwd_gemm_epilogue_gb300.tensor_parallel import TensorParallelSwiGLU
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        p = parts[rank]
        tp = TensorParallelSwiGLU(p["W1s"], p["W2s"], n_chunks=3, compute=_StoredCompute(p, rows))
        y, _ = tp.forward(p["x"])
        dx, _, _ = tp.backward(p["x"], p["pre"], p["dy"])
        out[rank] = (y.numpy(), dx.numpy())
    finally:
        dist.destroy_process_group()


def test_library_shard_outputs_reduced_by_two_gloo_ranks(b):
    # The library's shard outputs (fp32 copies on the host) go through the tensor-parallel
    # module's chunked all-reduce on two gloo ranks; every rank must end with the block's y, dx.
    import torch.multiprocessing as mp
    s = Shape(300, 256, 512, 264)
    _, x, W1, W2, dy = workloads.make_block(s, seed=93)
    p_ref, _, y_ref = oracle.fwd(x, W1, W2)
    pre = torch.from_numpy(p_ref).to(torch.bfloat16)
    _, _, _, dx_ref, _, _ = oracle.bwd_full(x, W1, W2, pre, dy)
    shards = run_shards(b, s, 2, x, W1, W2, dy, pre)
    parts = [{k: (v.float().cpu() if torch.is_tensor(v) else v) for k, v in o.items()} for o in shards]
    for p in parts:
        p.update(x=x.float(), dy=dy.float())
    with mp.get_context("spawn").Manager() as m:
        out = m.dict()
        mp.spawn(_gloo_rank, args=(2, _free_port(), parts, 128, out), nprocs=2, join=True)
        res = dict(out)
    for rank in range(2):
        parity(res[rank][0], y_ref, f"y on gloo rank {rank}")
        parity(res[rank][1], dx_ref, f"dx on gloo rank {rank}")


def test_shard_calls_capture_into_a_cuda_graph(b):
    # The chunked forward and the evented backward fork onto the library's second stream and
    # join back; captured into a CUDA graph, their replays give the direct calls' bits.
    s = Shape(1000, 256, 768, 320)
    _, x, W1, W2, dy = workloads.make_block(s, seed=98)
    xd, W1d, W2d, dyd = dev(x), dev(W1), dev(W2), dev(dy)
    j0, Hs = shard_bounds(s.H, 2, 1)
    W1s, W2s = b.swiglu_mlp_tp_shard_pack(W1d, W2d, j0, Hs)
    bf = dict(dtype=torch.bfloat16, device="cuda")
    pre, y = torch.empty(s.M, 2 * Hs, **bf), torch.empty(s.M, s.Dout, **bf)
    dx, dW1, dW2 = torch.empty(s.M, s.D, **bf), torch.empty(2 * Hs, s.D, **bf), torch.empty(s.Dout, Hs, **bf)
    wsf = torch.empty(b.swiglu_mlp_fwd_workspace_size(s.M, s.D, Hs, s.Dout), dtype=torch.uint8, device="cuda")
    wsb = torch.empty(b.swiglu_mlp_bwd_workspace_size(s.M, s.D, Hs, s.Dout), dtype=torch.uint8, device="cuda")
    events = [torch.cuda.Event() for _ in range(4)]
    ev = torch.cuda.Event()

    def step():
        b.swiglu_mlp_tp_fwd(xd, W1s, W2s, pre, y, wsf, n_chunks=4, chunk_events=events)
        b.swiglu_mlp_tp_bwd(xd, W1s, W2s, pre, dyd, dx, dW1, dW2, wsb, dx_event=ev)

    step()
    torch.cuda.synchronize()
    assert b.swiglu_mlp_device_status() == 0
    ref = [t.clone() for t in (pre, y, dx, dW1, dW2)]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="relaxed"):
        step()
    for t in (pre, y, dx, dW1, dW2):
        t.zero_()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert b.swiglu_mlp_device_status() == 0
    for name, got, want in zip(("preact", "y", "dx", "dW1", "dW2"), (pre, y, dx, dW1, dW2), ref):
        assert torch.equal(got, want), name
