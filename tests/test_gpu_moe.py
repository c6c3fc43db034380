"""GPU parity of the mixture-of-experts layer (swiglu_moe_fwd / swiglu_moe_bwd,
through the C ABI) against the fp64 CPU oracle.

Each expert is the SwiGLU block on its own rows with its own weights; the CUDA
path runs each step as one grouped launch over all experts.  Small cases are
compared over whole tensors and cover the edge cases of ragged grouping: experts
with no rows (first, middle, last), a single row, row counts just past a tile,
every row in one expert, many small experts (the 128-row tile choice).  The
named MoE workloads run at full size in the launch configuration the benchmark
times and are compared on sampled rows and on sampled hidden columns of a few
experts' weight gradients.
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


def dev(t):
    return t.cuda().contiguous()


def _experts(counts, D, H, Dout, seed):
    E, T = len(counts), sum(counts)
    s = Shape(T, D, H, Dout)
    x, dy = workloads.make_activations(s, seed)
    W1 = workloads.normal_bf16((E, 2 * H, D), D ** -0.5, seed, 1)
    W2 = workloads.normal_bf16((E, Dout, H), H ** -0.5, seed, 2)
    preact = workloads.make_preact(s, seed, gate_sweep=True)
    return x, W1, W2, dy, preact


CASES = {
    "pages_counts": ([32, 120, 8, 64], 256, 512, 256),
    "ragged": ([0, 300, 1, 129, 77, 0], 264, 392, 136),
    "one_expert": ([0, 0, 517, 0], 128, 256, 192),
    "many_small": ([3, 0, 17, 40, 64, 1, 0, 90, 33, 12, 5, 71, 0, 128, 2, 9], 128, 200, 128),
}


@pytest.fixture(params=["default", "single"])
def moe_cta(request, b):
    b.swiglu_mlp_set_debug_flags(2 if request.param == "single" else 0)
    yield request.param
    b.swiglu_mlp_set_debug_flags(0)


@pytest.mark.parametrize("case", list(CASES))
def test_moe_forward_matches_oracle(b, moe_cta, case):
    counts, D, H, Dout = CASES[case]
    x, W1, W2, _, _ = _experts(counts, D, H, Dout, seed=80)
    p_ref, _, y_ref = oracle.moe_fwd(x, W1, W2, counts)
    preact, y = b.swiglu_moe_fwd(dev(x), dev(W1), dev(W2), counts)
    assert b.swiglu_mlp_device_status() == 0
    parity(preact, p_ref, f"preact ({case})")
    parity(y, y_ref, f"y ({case})")


@pytest.fixture(params=["grouped", "ungrouped", "single"])
def moe_bwd_mode(request, b):
    b.swiglu_mlp_set_debug_flags({"grouped": 0, "ungrouped": 4, "single": 2}[request.param])
    yield request.param
    b.swiglu_mlp_set_debug_flags(0)


@pytest.mark.parametrize("case", list(CASES))
def test_moe_backward_matches_oracle(b, moe_bwd_mode, case):
    counts, D, H, Dout = CASES[case]
    x, W1, W2, dy, preact = _experts(counts, D, H, Dout, seed=81)
    _, gp_ref, h_ref, dx_ref, dW1_ref, dW2_ref = oracle.moe_bwd_full(x, W1, W2, preact, dy, counts)
    T = sum(counts)
    ws = torch.empty(b.swiglu_moe_bwd_workspace_size(counts, D, H, Dout), dtype=torch.uint8, device="cuda")
    # poison the outputs: an expert without rows must still get zero weight gradients
    dW1 = torch.full((len(counts), 2 * H, D), 3.0, dtype=torch.bfloat16, device="cuda")
    dW2 = torch.full((len(counts), Dout, H), 3.0, dtype=torch.bfloat16, device="cuda")
    dx, dW1, dW2 = b.swiglu_moe_bwd(dev(x), dev(W1), dev(W2), dev(preact), dev(dy), counts,
                                    dW1=dW1, dW2=dW2, workspace=ws)
    assert b.swiglu_mlp_device_status() == 0
    h, gp = b.bwd_workspace_views(ws, T, H)
    parity(gp, gp_ref, "grad_preact")
    parity(h, h_ref, "h")
    parity(dx, dx_ref, "dx")
    for e in range(len(counts)):
        if counts[e] == 0:
            assert dW1[e].abs().max().item() == 0 and dW2[e].abs().max().item() == 0
        else:
            parity(dW1[e], dW1_ref[e], f"dW1[{e}]")
            parity(dW2[e], dW2_ref[e], f"dW2[{e}]")


def test_moe_no_rows(b):
    counts = [0, 0, 0]
    E, D, H, Dout = 3, 64, 128, 64
    W1 = dev(workloads.normal_bf16((E, 2 * H, D), 0.1, 82, 1))
    W2 = dev(workloads.normal_bf16((E, Dout, H), 0.1, 82, 2))
    x = torch.empty(0, D, dtype=torch.bfloat16, device="cuda")
    preact, y = b.swiglu_moe_fwd(x, W1, W2, counts)
    assert preact.shape == (0, 2 * H) and y.shape == (0, Dout)
    dW1 = torch.full((E, 2 * H, D), 5.0, dtype=torch.bfloat16, device="cuda")
    dW2 = torch.full((E, Dout, H), 5.0, dtype=torch.bfloat16, device="cuda")
    _, dW1, dW2 = b.swiglu_moe_bwd(x, W1, W2, preact, torch.empty(0, Dout, dtype=torch.bfloat16, device="cuda"),
                                   counts, dW1=dW1, dW2=dW2)
    assert b.swiglu_mlp_device_status() == 0
    assert dW1.abs().max().item() == 0 and dW2.abs().max().item() == 0


def _sample(n, k, seed):
    rng = np.random.default_rng(seed)
    idx = rng.choice(n, size=min(k, n), replace=False)
    return np.unique(np.concatenate([idx, [0, n - 1]]))


@pytest.mark.parametrize("name", ["moe8", "moe64"])
def test_moe_full_size_sampled(b, name):
    counts, x, W1, W2, dy = workloads.make_moe(name)
    E, D, H, Dout = W1.shape[0], x.shape[1], W2.shape[2], W2.shape[1]
    T = sum(counts)
    cfg = workloads.MOE_CONFIGS[name]
    preact_in = workloads.make_preact(Shape(T, D, H, Dout), cfg["seed"])
    xd, W1d, W2d, dyd, prd = dev(x), dev(W1), dev(W2), dev(dy), dev(preact_in)
    preact, y = b.swiglu_moe_fwd(xd, W1d, W2d, counts)
    ws = torch.empty(b.swiglu_moe_bwd_workspace_size(counts, D, H, Dout), dtype=torch.uint8, device="cuda")
    dx, dW1, dW2 = b.swiglu_moe_bwd(xd, W1d, W2d, prd, dyd, counts, workspace=ws)
    assert b.swiglu_mlp_device_status() == 0
    h, gp = b.bwd_workspace_views(ws, T, H)

    off = oracle.expert_offsets(counts)
    # the first and last row of every third expert with rows, plus random rows
    edges = [v for e in range(0, E, 3) if counts[e] for v in (off[e], off[e + 1] - 1)]
    rows = np.unique(np.concatenate([_sample(T, 6, 4), edges]))
    p_fwd, y_ref, gp_ref, h_ref, dx_ref = oracle.moe_rows(x, W1, W2, preact_in, dy, counts, rows)
    parity(preact[rows], p_fwd, "preact[rows]")
    parity(y[rows], y_ref, "y[rows]")
    parity(gp[rows], gp_ref, "grad_preact[rows]")
    parity(h[rows], h_ref, "h[rows]")
    parity(dx[rows], dx_ref, "dx[rows]")
    cols = _sample(H, 3, 5)
    for e in [0, E // 2, E - 1]:
        dW2c, dW1l, dW1g = oracle.moe_cols(x, W2, preact_in, dy, counts, e, cols)
        parity(dW2[e][:, cols].T, dW2c, f"dW2[{e}][:, cols]")
        parity(dW1[e][cols], dW1l, f"dW1[{e}][cols]")
        parity(dW1[e][H + cols], dW1g, f"dW1[{e}][H + cols]")


def test_moe_host_step_runner_matches_direct_calls(b):
    # the overlapped host-batch runner gives the same bits as direct calls
    from bwd_gemm_epilogue_gb300.pipeline import HostStepRunner
    counts, D, H, Dout = CASES["ragged"]
    x, W1, W2, dy, _ = _experts(counts, D, H, Dout, seed=83)
    T = sum(counts)
    preact, y = b.swiglu_moe_fwd(dev(x), dev(W1), dev(W2), counts)
    dx, dW1, dW2 = b.swiglu_moe_bwd(dev(x), dev(W1), dev(W2), preact, dev(dy), counts)
    r = HostStepRunner(T, D, H, Dout, counts=counts)
    host_in = {k: t.pin_memory() for k, t in (("x", x), ("W1", W1), ("W2", W2), ("dy", dy))}
    outs = [{k: torch.empty(t.shape, dtype=t.dtype).pin_memory() for k, t in
             (("y", y), ("dx", dx), ("dW1", dW1), ("dW2", dW2))} for _ in range(3)]
    r.run([host_in] * 3, outs)
    r.synchronize()
    assert b.swiglu_mlp_device_status() == 0
    for o in outs:
        for k, ref in (("y", y), ("dx", dx), ("dW1", dW1), ("dW2", dW2)):
            assert torch.equal(o[k], ref.cpu()), k


def _random_moe(n, seed):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        E = int(rng.integers(1, 13))
        counts = [int(c) if rng.random() > 0.2 else 0 for c in rng.integers(0, 400, size=E)]
        D, H, Dout = (8 * int(rng.integers(1, 50)) for _ in range(3))
        out.append((counts, D, H, Dout))
    return out


@pytest.mark.parametrize("case", _random_moe(8, 77), ids=lambda c: f"E{len(c[0])}_T{sum(c[0])}_D{c[1]}_H{c[2]}")
def test_moe_random_layers(b, case):
    counts, D, H, Dout = case
    x, W1, W2, dy, preact = _experts(counts, D, H, Dout, seed=84 + len(counts))
    p_ref, _, y_ref = oracle.moe_fwd(x, W1, W2, counts)
    _, gp_ref, _, dx_ref, dW1_ref, dW2_ref = oracle.moe_bwd_full(x, W1, W2, preact, dy, counts)
    T = sum(counts)
    ws = torch.empty(max(16, b.swiglu_moe_bwd_workspace_size(counts, D, H, Dout)), dtype=torch.uint8, device="cuda")
    pre_gpu, y = b.swiglu_moe_fwd(dev(x), dev(W1), dev(W2), counts)
    dx, dW1, dW2 = b.swiglu_moe_bwd(dev(x), dev(W1), dev(W2), dev(preact), dev(dy), counts, workspace=ws)
    assert b.swiglu_mlp_device_status() == 0
    if T:
        parity(pre_gpu, p_ref, "preact")
        parity(y, y_ref, "y")
        parity(b.bwd_workspace_views(ws, T, H)[1], gp_ref, "grad_preact")
        parity(dx, dx_ref, "dx")
    for e in range(len(counts)):
        if counts[e]:
            parity(dW1[e], dW1_ref[e], f"dW1[{e}]")
            parity(dW2[e], dW2_ref[e], f"dW2[{e}]")
        else:
            assert dW1[e].abs().max().item() == 0 and dW2[e].abs().max().item() == 0


def test_moe_many_calls_in_flight(b):
    # 20 forward calls queued back to back (more than the 8 pinned table slots, each call
    # copying two tables) on two streams, with different counts and inputs per call; every
    # result must be the one its own call asked for
    D, H, Dout = 64, 128, 64
    calls = []
    for i in range(20):
        counts = [(7 * i + 3 * e) % 50 for e in range(3)]
        x, W1, W2, _, _ = _experts(counts, D, H, Dout, seed=200 + i)
        calls.append((counts, x, W1, W2))
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = []
    for i, (counts, x, W1, W2) in enumerate(calls):
        with torch.cuda.stream(streams[i % 2]):
            outs.append(b.swiglu_moe_fwd(dev(x), dev(W1), dev(W2), counts))
    torch.cuda.synchronize()
    assert b.swiglu_mlp_device_status() == 0
    for (counts, x, W1, W2), (_, y) in zip(calls, outs):
        if sum(counts):
            parity(y, oracle.moe_fwd(x, W1, W2, counts)[2], f"y (counts {counts})")
