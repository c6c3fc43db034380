"""256 x 512 tiles (two TMEM accumulator slots per CTA-pair tile) against 256 x 256 tiles.

Both tile shapes accumulate every output element over the same k-steps in the same order
with the same MMA shape (M = 256, N = 256, K = 16), so their results must agree bit for
bit; the wide tiles are also checked against the fp64 product and the oracle.  The test
hook bits force one tile shape (32: 256 x 256 everywhere, 64: 256 x 512 wherever N > 256)
instead of the library's choice.
"""
import pytest
import torch

import oracle
from bwd_gemm_epilogue_gb300 import workloads
from bwd_gemm_epilogue_gb300.workloads import Shape
from helpers import ensure_library, parity

pytestmark = pytest.mark.gpu
NARROW, WIDE = 32, 64


@pytest.fixture(scope="module")
def b():
    ensure_library()
    from bwd_gemm_epilogue_gb300 import binding
    binding.lib()
    yield binding
    binding.swiglu_mlp_set_debug_flags(0)


def dev(t):
    return t.cuda().contiguous()


def with_flags(b, flags, fn):
    b.swiglu_mlp_set_debug_flags(flags)
    try:
        out = fn()
        torch.cuda.synchronize()
    finally:
        b.swiglu_mlp_set_debug_flags(0)
    assert b.swiglu_mlp_device_status() == 0
    return out


# N values: whole 512-column tiles, a last tile with only its first slot (N = 768, 1280),
# a second slot of 8 columns (N = 264, 520 + 8), and M that ends inside a CTA pair's rows
# (M a multiple of 8: MN-major A has M contiguous).
GEMMS = [(296, 520, 200), (512, 768, 1000), (1000, 1024, 64), (304, 264, 8), (264, 2056, 136), (640, 1280, 4096)]


@pytest.mark.parametrize("a_mn,b_mn", [(False, False), (False, True), (True, True), (True, False)])
@pytest.mark.parametrize("M,N,K", GEMMS, ids=lambda v: str(v))
def test_wide_tiles_equal_narrow_tiles(b, a_mn, b_mn, M, N, K):
    g = torch.Generator().manual_seed(M + 3 * N + 7 * K)
    A = torch.randn(M, K, generator=g).to(torch.bfloat16)
    B = torch.randn(N, K, generator=g).to(torch.bfloat16)
    A_in = dev(A.T.contiguous() if a_mn else A)
    B_in = dev(B.T.contiguous() if b_mn else B)
    run = lambda: b.swiglu_mlp_gemm_bf16(A_in, B_in, M, N, K, a_mn, b_mn)
    c_narrow = with_flags(b, NARROW, run)
    c_wide = with_flags(b, WIDE, run)
    assert torch.equal(c_narrow, c_wide)
    parity(c_wide, (A.double() @ B.double().T).numpy(), f"C wide a_mn={a_mn} b_mn={b_mn}")


@pytest.mark.parametrize("s", [Shape(300, 256, 520, 264), Shape(640, 128, 1024, 768), Shape(1000, 256, 768, 320)],
                         ids=lambda s: f"M{s.M}_D{s.D}_H{s.H}_Do{s.Dout}")
def test_block_with_wide_tiles_matches_oracle_and_narrow_bits(b, s):
    _, x, W1, W2, dy = workloads.make_block(s, seed=61)
    p_ref, _, y_ref = oracle.fwd(x, W1, W2)
    pre = torch.from_numpy(p_ref).to(torch.bfloat16)
    _, gp_ref, _, dx_ref, dW1_ref, dW2_ref = oracle.bwd_full(x, W1, W2, pre, dy)
    xd, W1d, W2d, dyd, pred = dev(x), dev(W1), dev(W2), dev(dy), dev(pre)
    res = {}
    for name, flags in (("narrow", NARROW), ("wide", WIDE), ("wide, three launches", WIDE | 4)):
        fwd = with_flags(b, flags, lambda: b.swiglu_mlp_fwd(xd, W1d, W2d))
        bwd = with_flags(b, flags, lambda: b.swiglu_mlp_bwd(xd, W1d, W2d, pred, dyd))
        res[name] = fwd + bwd
    for name in ("wide", "wide, three launches"):
        for u, v, what in zip(res["narrow"], res[name], ("preact", "y", "dx", "dW1", "dW2")):
            assert torch.equal(u, v), f"{what}: {name} tiles differ from narrow tiles"
    _, y, dx, dW1, dW2 = res["wide"]
    parity(y, y_ref, "y (wide down projection)")
    parity(dx, dx_ref, "dx")
    parity(dW1, dW1_ref, "dW1")
    parity(dW2, dW2_ref, "dW2")


@pytest.mark.parametrize("s", [Shape(300, 256, 520, 256), Shape(1000, 256, 768, 256)],
                         ids=lambda s: f"M{s.M}_D{s.D}_H{s.H}")
def test_residual_block_with_wide_tiles(b, s):
    # The residual block: its backward group adds dy into dx in the residual epilogue, in
    # 256 x 512 tiles when forced (the single residual down projection keeps 256 x 256).
    _, x, W1, W2, dy = workloads.make_block(s, seed=62)
    p_ref, _, y_ref = oracle.fwd(x, W1, W2, residual=True)
    pre = torch.from_numpy(p_ref).to(torch.bfloat16)
    _, _, _, dx_ref, dW1_ref, dW2_ref = oracle.bwd_full(x, W1, W2, pre, dy, residual=True)
    xd, W1d, W2d, dyd, pred = dev(x), dev(W1), dev(W2), dev(dy), dev(pre)
    res = {}
    for name, flags in (("narrow", NARROW), ("wide", WIDE), ("wide, three launches", WIDE | 4)):
        fwd = with_flags(b, flags, lambda: b.swiglu_mlp_fwd(xd, W1d, W2d, residual=True))
        bwd = with_flags(b, flags, lambda: b.swiglu_mlp_bwd(xd, W1d, W2d, pred, dyd, residual=True))
        res[name] = fwd + bwd
    for name in ("wide", "wide, three launches"):
        for u, v, what in zip(res["narrow"], res[name], ("preact", "y", "dx", "dW1", "dW2")):
            assert torch.equal(u, v), f"{what} (residual): {name} tiles differ from narrow tiles"
    _, y, dx, dW1, dW2 = res["wide"]
    parity(y, y_ref, "y (residual)")
    parity(dx, dx_ref, "dx (residual, wide tiles)")
    parity(dW1, dW1_ref, "dW1 (residual block, wide tiles)")
    parity(dW2, dW2_ref, "dW2 (residual block, wide tiles)")


def test_wide_tile_wait_times_out_and_context_survives(b):
    A = torch.randn(512, 128).to(torch.bfloat16).cuda()
    B = torch.randn(768, 128).to(torch.bfloat16).cuda()
    b.swiglu_mlp_set_wait_timeout_ns(50_000_000)
    b.swiglu_mlp_set_debug_flags(1 | WIDE)   # producer issues nothing: every consumer wait runs out
    try:
        b.swiglu_mlp_gemm_bf16(A, B, 512, 768, 128, False, False)
        assert b.swiglu_mlp_device_status() == 6      # SWIGLU_ERR_TIMEOUT
    finally:
        b.swiglu_mlp_set_debug_flags(0)
        b.swiglu_mlp_set_wait_timeout_ns(4_000_000_000)
    assert b.swiglu_mlp_device_status() == 0
    C = with_flags(b, WIDE, lambda: b.swiglu_mlp_gemm_bf16(A, B, 512, 768, 128, False, False))
    parity(C, (A.double() @ B.double().T).cpu().numpy(), "C after timeout")


@pytest.mark.parametrize("case", ["pages_counts", "ragged", "one_expert", "many_small"])
def test_moe_layer_with_wide_tiles_matches_narrow_bits(b, case):
    # the experts' down projections and weight-gradient / dx products in one table launch
    from test_gpu_moe import CASES, _experts
    counts, D, H, Dout = CASES[case]
    x, W1, W2, dy, preact = _experts(counts, D, H, Dout, seed=83)
    xd, W1d, W2d, dyd, pred = dev(x), dev(W1), dev(W2), dev(dy), dev(preact)
    res = {}
    for name, flags in (("narrow", NARROW), ("wide", WIDE), ("wide, three launches", WIDE | 4)):
        fwd = with_flags(b, flags, lambda: b.swiglu_moe_fwd(xd, W1d, W2d, counts))
        bwd = with_flags(b, flags, lambda: b.swiglu_moe_bwd(xd, W1d, W2d, pred, dyd, counts))
        res[name] = fwd + bwd
    for name in ("wide", "wide, three launches"):
        for u, v, what in zip(res["narrow"], res[name], ("preact", "y", "dx", "dW1", "dW2")):
            assert torch.equal(u, v), f"{what}: {name} tiles differ from narrow tiles ({case})"
    y_ref = oracle.moe_fwd(x, W1, W2, counts)[2]
    parity(res["wide"][1], y_ref, f"y, wide tiles ({case})")
    _, _, _, dx_ref, dW1_ref, dW2_ref = oracle.moe_bwd_full(x, W1, W2, preact, dy, counts)
    parity(res["wide"][2], dx_ref, f"dx, wide tiles ({case})")
    for e in range(len(counts)):
        if counts[e]:
            parity(res["wide"][3][e], dW1_ref[e], f"dW1[{e}], wide tiles ({case})")
            parity(res["wide"][4][e], dW2_ref[e], f"dW2[{e}], wide tiles ({case})")


@pytest.mark.parametrize("M,N,K", [(5568, 3584, 7168), (11136, 3584, 14336), (2816, 3848, 6400)], ids=lambda v: str(v))
def test_mixed_tile_widths_in_one_launch(b, M, N, K):
    # A long-K product with few 256 x 512 tiles per CTA pair: the library keeps its first rows
    # in 256 x 512 tiles and runs the last row tiles as 256 x 256 tiles in the same launch
    # (for these shapes: rows 0..5375 / 0..11007 / 0..2303 wide; the last N ends 8 columns into a
    # tile's second slot and into a 256 x 256 tile).  Bits as with 256 x 256 tiles only,
    # rows on both sides of the split against the fp64 product.
    g = torch.Generator().manual_seed(M + N + K)
    A = (torch.randn(M, K, generator=g) * K ** -0.25).to(torch.bfloat16)
    B = (torch.randn(N, K, generator=g) * K ** -0.25).to(torch.bfloat16)
    Ad, Bd = dev(A), dev(B)
    c_auto = with_flags(b, 0, lambda: b.swiglu_mlp_gemm_bf16(Ad, Bd, M, N, K, False, False))
    c_narrow = with_flags(b, NARROW, lambda: b.swiglu_mlp_gemm_bf16(Ad, Bd, M, N, K, False, False))
    assert torch.equal(c_auto, c_narrow)
    split = {5568: 5376, 11136: 11008, 2816: 2304}[M]
    rows = torch.tensor(sorted({0, 255, 256, split - 257, split - 1, split, split + 1, M - 1, M // 2}))
    ref = A[rows].double() @ B.double().T
    parity(c_auto[rows.cuda()], ref.numpy(), "C rows around the split")
