"""GPU parity of the FP8 forward (swiglu_mlp_fwd_fp8, through the C ABI) against
the fp64 CPU oracle.

preact and y are compared with the floating-point bar.  h8 is an integer code
decided by floating point: where the oracle's h / s_h lies close to the midpoint
between two E4M3 codes (closer than the GPU's fp32 arithmetic -- MUFU sigmoid,
fp32 scale products -- can resolve), either neighbour is valid; everywhere else
the codes must be equal.  Saturation at +-448 is checked the same way.
"""
import numpy as np
import pytest
import torch

import oracle
from bwd_gemm_epilogue_gb300 import workloads
from bwd_gemm_epilogue_gb300.workloads import Shape
from helpers import ensure_library, parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def b():
    ensure_library()
    from bwd_gemm_epilogue_gb300 import binding
    binding.lib()
    return binding


@pytest.fixture(params=["pair", "single"])
def cta_mode(request, b):
    b.swiglu_mlp_set_debug_flags(2 if request.param == "single" else 0)
    yield request.param
    b.swiglu_mlp_set_debug_flags(0)


_LUT = np.array([oracle.e4m3_decode(c) for c in range(256)])


def check_codes(h8_gpu, hpre, h8_ref, s_h, what):
    got = h8_gpu.view(torch.uint8).cpu().numpy().astype(np.int64)
    ref = h8_ref.astype(np.int64)
    q = hpre / s_h
    dg = _LUT[got]
    assert not np.isnan(dg).any(), f"{what}: NaN code"
    a = np.abs(q)
    spacing = np.where(a < 2.0 ** -6, 2.0 ** -9, 2.0 ** (np.floor(np.log2(np.maximum(a, 2.0 ** -6))) - 3))
    slack = spacing / 2 + 2.0 ** -7 * a                    # a neighbour within the GPU's resolution
    ok = (got == ref) | (np.abs(dg - np.clip(q, -448, 448)) <= slack)
    assert ok.all(), f"{what}: {int((~ok).sum())} codes off by more than one step"
    mism = float((got != ref).mean())
    assert mism < 0.01, f"{what}: {mism:.4f} of the codes differ from the oracle's"
    return mism


SHAPES = [Shape(128, 256, 512, 256), Shape(300, 320, 400, 264), Shape(1, 64, 128, 72), Shape(520, 128, 272, 136)]


@pytest.mark.parametrize("s", SHAPES, ids=lambda s: f"M{s.M}_D{s.D}_H{s.H}_Do{s.Dout}")
def test_fp8_forward_matches_oracle(b, cta_mode, s):
    x8, W1_8, W2_8, sc = workloads.make_fp8_block(s, seed=91, s_h=1.0 / 128)   # saturates above 3.5
    p_ref, hpre, h8_ref, y_ref = oracle.fwd_fp8(x8, W1_8, W2_8, **sc)
    preact, h8, y = b.swiglu_mlp_fwd_fp8(x8.cuda(), W1_8.cuda(), W2_8.cuda(), **sc)
    assert b.swiglu_mlp_device_status() == 0
    parity(preact, p_ref, "preact")
    check_codes(h8, hpre, h8_ref, sc["s_h"], "h8")
    parity(y, y_ref, "y")


def test_fp8_forward_without_preact_and_saturation(b):
    s = Shape(256, 128, 256, 128)
    x8, W1_8, W2_8, sc = workloads.make_fp8_block(s, seed=92, s_h=1.0 / 1024)  # many saturate
    _, hpre, h8_ref, y_ref = oracle.fwd_fp8(x8, W1_8, W2_8, **sc)
    pre, h8, y = b.swiglu_mlp_fwd_fp8(x8.cuda(), W1_8.cuda(), W2_8.cuda(), store_preact=False, **sc)
    assert pre is None and b.swiglu_mlp_device_status() == 0
    codes = h8.view(torch.uint8).cpu().numpy()
    assert ((codes & 0x7F) == 0x7E).mean() > 0.05       # a good share saturated at +-448
    check_codes(h8, hpre, h8_ref, sc["s_h"], "h8 (saturating)")
    parity(y, y_ref, "y")


def test_fp8_forward_full_size_sampled(b):
    # the 4096-token LLaMA-7B-shaped block in FP8, compared on sampled rows
    s = workloads.CONFIGS["prefill"]["shape"]
    x8, W1_8, W2_8, sc = workloads.make_fp8_block(s, seed=2)
    preact, h8, y = b.swiglu_mlp_fwd_fp8(x8.cuda(), W1_8.cuda(), W2_8.cuda(), **sc)
    assert b.swiglu_mlp_device_status() == 0
    rows = np.array([0, 1, 777, 2048, 4095])
    p_ref, hpre, h8_ref, y_ref = oracle.fwd_fp8(x8, W1_8, W2_8, rows=rows, **sc)
    parity(preact[rows], p_ref, "preact[rows]")
    check_codes(h8[rows], hpre, h8_ref, sc["s_h"], "h8[rows]")
    parity(y[rows], y_ref, "y[rows]")


@pytest.mark.parametrize("M", [1, 16, 40, 64])
@pytest.mark.parametrize("small_m_path", [True, False])
def test_fp8_few_tokens(b, M, small_m_path):
    # M <= 64: the FP8 weights stream through the transposed, K-split kernels (the
    # decode path); test hook bit 3 keeps the 128/256-row tile kernels for comparison
    s = Shape(M, 512, 1024, 768)
    x8, W1_8, W2_8, sc = workloads.make_fp8_block(s, seed=93 + M, s_h=1.0 / 128)
    p_ref, hpre, h8_ref, y_ref = oracle.fwd_fp8(x8, W1_8, W2_8, **sc)
    b.swiglu_mlp_set_debug_flags(0 if small_m_path else 8)
    try:
        preact, h8, y = b.swiglu_mlp_fwd_fp8(x8.cuda(), W1_8.cuda(), W2_8.cuda(), **sc)
        assert b.swiglu_mlp_device_status() == 0
    finally:
        b.swiglu_mlp_set_debug_flags(0)
    parity(preact, p_ref, "preact")
    check_codes(h8, hpre, h8_ref, sc["s_h"], "h8")
    parity(y, y_ref, "y")


def _random_fp8_shapes(n, seed):
    rng = np.random.default_rng(seed)
    return [Shape(int(rng.choice([int(rng.integers(1, 65)), int(rng.integers(65, 600))])),
                  16 * int(rng.integers(1, 40)), 16 * int(rng.integers(1, 40)), 8 * int(rng.integers(1, 80)))
            for _ in range(n)]


@pytest.mark.parametrize("s", _random_fp8_shapes(10, 31), ids=lambda s: f"M{s.M}_D{s.D}_H{s.H}_Do{s.Dout}")
def test_fp8_random_shapes(b, s):
    x8, W1_8, W2_8, sc = workloads.make_fp8_block(s, seed=95 + s.M, s_h=1.0 / 128)
    p_ref, hpre, h8_ref, y_ref = oracle.fwd_fp8(x8, W1_8, W2_8, **sc)
    preact, h8, y = b.swiglu_mlp_fwd_fp8(x8.cuda(), W1_8.cuda(), W2_8.cuda(), **sc)
    assert b.swiglu_mlp_device_status() == 0
    parity(preact, p_ref, "preact")
    check_codes(h8, hpre, h8_ref, sc["s_h"], "h8")
    parity(y, y_ref, "y")
