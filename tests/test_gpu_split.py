"""Split tiles of the forward's down projection y = h @ W2^T (256 x 512 tiles).

Where the last round of whole tiles would leave CTA pairs idle, the k-blocks of the last
tiles are divided evenly over the pairs, and a tile cut by a boundary is summed by two
pairs in fp32 and added once (tests/test_split_plan.py checks the lists on the host).
These tests run shapes whose forward splits tiles: y against the oracle in rows of every
M-tile, against the unsplit launch (test hook bit 7) to within the rounding of one extra
fp32 addition, bit-identical from run to run, and the bounded waits with split tiles.
"""
import numpy as np
import pytest
import torch

import oracle
from bwd_gemm_epilogue_gb300 import workloads
from bwd_gemm_epilogue_gb300.workloads import Shape
from helpers import TILE_REL_FRO, ensure_library, parity

pytestmark = pytest.mark.gpu
NO_SPLIT, SKIP_PRODUCER = 128, 1

# 160 tiles (one whole round, then 84 tiles' k-blocks shared, 100 k-blocks per tile);
# ragged rows (the last row tile ends inside a CTA pair) with 24 x 10 tiles; 16 x 16 tiles
# (four raster bands of column tiles, the tail crossing bands)
SHAPES = [Shape(5120, 256, 6400, 4096), Shape(6000, 512, 7168, 5120), Shape(4096, 512, 8192, 8192)]


@pytest.fixture(scope="module")
def b():
    ensure_library()
    from bwd_gemm_epilogue_gb300 import binding
    binding.lib()
    yield binding
    binding.swiglu_mlp_set_debug_flags(0)


def dev(t):
    return t.cuda().contiguous()


def ok_status(b):
    torch.cuda.synchronize()
    assert b.swiglu_mlp_device_status() == 0


def tile_rows(M, seed):
    rng = np.random.default_rng(seed)
    out = []
    for r0 in range(0, M, 128):   # every CTA's rows of every 256-row tile
        r1 = min(M, r0 + 128)
        out += [r0, r1 - 1, int(rng.integers(r0, r1))]
    return np.unique(np.asarray(out, dtype=np.int64))


def forward(b, x, W1, W2, flags=0, residual=False):
    b.swiglu_mlp_set_debug_flags(flags)
    try:
        _, y = b.swiglu_mlp_fwd(x, W1, W2, residual=residual)
        ok_status(b)
    finally:
        b.swiglu_mlp_set_debug_flags(0)
    return y


def close_to_unsplit(y, y_ref):
    # one more fp32 addition per element of a split tile: the bf16 outputs agree but for
    # rare last-bit roundings
    d = (y.float() - y_ref.float()).abs()
    scale = y_ref.float().abs().max().item()
    assert d.max().item() <= 2.0 ** -6 * scale
    assert (d > 0).float().mean().item() < 0.01
    assert torch.linalg.norm(d) <= 1e-3 * torch.linalg.norm(y_ref.float())


@pytest.mark.parametrize("s", SHAPES, ids=str)
def test_split_tiles_match_oracle(b, s):
    assert b.swiglu_mlp_split_plan(s.M, s.Dout, s.H, 76) is not None
    _, x, W1, W2, _ = workloads.make_block(s, seed=61)
    xd, W1d, W2d = dev(x), dev(W1), dev(W2)
    y = forward(b, xd, W1d, W2d)
    rows = tile_rows(s.M, 62)
    _, _, y_ref = oracle.fwd(x, W1, W2, rows=rows)
    parity(y[rows], y_ref, "y[rows]")
    for t in np.unique(rows // 256):
        r = rows[rows // 256 == t]
        k = np.searchsorted(rows, r)
        parity(y[r], y_ref[k], f"y rows of M-tile {t}", rel_fro=TILE_REL_FRO)
    close_to_unsplit(y, forward(b, xd, W1d, W2d, NO_SPLIT))


@pytest.mark.parametrize("residual", [False, True], ids=["plain", "residual"])
def test_split_tiles_full_size_against_unsplit_and_reproducible(b, residual):
    s, x, W1, W2, _ = workloads.make_block("target")
    assert b.swiglu_mlp_split_plan(s.M, s.Dout, s.H, 76) is not None
    xd, W1d, W2d = dev(x), dev(W1), dev(W2)
    y1 = forward(b, xd, W1d, W2d, residual=residual)
    y2 = forward(b, xd, W1d, W2d, residual=residual)
    assert torch.equal(y1, y2)   # which piece of a split tile arrives first does not matter
    close_to_unsplit(y1, forward(b, xd, W1d, W2d, NO_SPLIT, residual=residual))


def test_split_tiles_residual_block_matches_oracle(b):
    # y = x + h @ W2^T with the residual added once, in fp32, by the piece that stores the tile
    s = Shape(5120, 4096, 6400, 4096)
    assert b.swiglu_mlp_split_plan(s.M, s.Dout, s.H, 76) is not None
    _, x, W1, W2, _ = workloads.make_block(s, seed=64)
    xd, W1d, W2d = dev(x), dev(W1), dev(W2)
    y = forward(b, xd, W1d, W2d, residual=True)
    rows = tile_rows(s.M, 65)
    _, _, y_ref = oracle.fwd(x, W1, W2, rows=rows, residual=True)
    parity(y[rows], y_ref, "y[rows] (residual)")
    for t in np.unique(rows // 256):
        r = rows[rows // 256 == t]
        k = np.searchsorted(rows, r)
        parity(y[r], y_ref[k], f"residual y rows of M-tile {t}", rel_fro=TILE_REL_FRO)
    close_to_unsplit(y, forward(b, xd, W1d, W2d, NO_SPLIT, residual=True))


def test_split_launch_times_out_and_recovers(b):
    s = SHAPES[0]
    _, x, W1, W2, _ = workloads.make_block(s, seed=63)
    xd, W1d, W2d = dev(x), dev(W1), dev(W2)
    ref = forward(b, xd, W1d, W2d)
    b.swiglu_mlp_set_wait_timeout_ns(50_000_000)
    b.swiglu_mlp_set_debug_flags(SKIP_PRODUCER)   # no loads: every consumer wait runs out
    try:
        b.swiglu_mlp_fwd(xd, W1d, W2d)
        assert b.swiglu_mlp_device_status() == 6  # SWIGLU_ERR_TIMEOUT
    finally:
        b.swiglu_mlp_set_debug_flags(0)
        b.swiglu_mlp_set_wait_timeout_ns(4_000_000_000)
    assert b.swiglu_mlp_device_status() == 0
    assert torch.equal(forward(b, xd, W1d, W2d), ref)


def test_split_forward_in_a_cuda_graph_and_on_two_streams(b):
    # the split launch enqueues a memset of its counters and the kernel on the caller's
    # stream: a CUDA graph replays it with the direct call's bits, and forwards on two
    # streams with their own workspaces (their own counters and sums) do not interfere
    s = SHAPES[0]
    _, x, W1, W2, _ = workloads.make_block(s, seed=66)
    xd, W1d, W2d = dev(x), dev(W1), dev(W2)
    x2 = dev(workloads.make_block(s, seed=67)[1])
    ref = forward(b, xd, W1d, W2d)
    ref2 = forward(b, x2, W1d, W2d)
    bf = dict(dtype=torch.bfloat16, device="cuda")
    preact, y = torch.empty(s.M, 2 * s.H, **bf), torch.empty(s.M, s.Dout, **bf)
    ws = torch.empty(b.swiglu_mlp_fwd_workspace_size(s.M, s.D, s.H, s.Dout), dtype=torch.uint8, device="cuda")
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        b.swiglu_mlp_fwd(xd, W1d, W2d, preact, y, ws)
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="relaxed"):
        b.swiglu_mlp_fwd(xd, W1d, W2d, preact, y, ws)
    y.zero_()
    g.replay()
    g.replay()
    ok_status(b)
    assert torch.equal(y, ref)

    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = []
    for st in streams:
        st.wait_stream(torch.cuda.current_stream())
    for _ in range(3):
        outs = []
        for st, xi in zip(streams, (xd, x2)):
            with torch.cuda.stream(st):
                outs.append(b.swiglu_mlp_fwd(xi, W1d, W2d)[1])
        for st in streams:
            torch.cuda.current_stream().wait_stream(st)
        ok_status(b)
        assert torch.equal(outs[0], ref) and torch.equal(outs[1], ref2)
