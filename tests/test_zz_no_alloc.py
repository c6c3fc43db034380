"""The allocation-free forward (swiglu_mlp_fwd_noalloc) against the ordinary one.

swiglu_mlp_fwd_noalloc serves callers that cannot allocate device memory (a
plugin whose host framework owns all allocations, a real-time loop that must
not call cudaMalloc, a process with a fixed memory budget): it keeps the
forward's transient h in a 64 MiB array built into the library instead of a
caller workspace.  Its results must be swiglu_mlp_fwd's bits where both run the
same kernels (M > 64), must match the oracle where they do not (M <= 64), and a
second call must not be disturbed by what the first one left in that shared
array.

The file name sorts last so that a run stopping at the first failure has
already run every other test; it also passes when run alone in a new process.
"""
import ctypes

import pytest
import torch

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


def _noalloc_via_abi(b, x, W1, W2):
    """Call the C entry point directly with plain device pointers."""
    M, D = x.shape
    H, Dout = W2.shape[1], W2.shape[0]
    preact = torch.empty(M, 2 * H, dtype=torch.bfloat16, device=x.device)
    y = torch.empty(M, Dout, dtype=torch.bfloat16, device=x.device)
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = b.lib().swiglu_mlp_fwd_noalloc(p(x), p(W1), p(W2), p(preact), p(y), M, D, H, Dout, stream)
    assert st == 0, b.lib().swiglu_mlp_last_error_detail()
    return preact, y


@pytest.mark.parametrize("s", [Shape(300, 320, 392, 264), Shape(1024, 512, 1536, 768)],
                         ids=lambda s: f"M{s.M}_D{s.D}_H{s.H}_Do{s.Dout}")
def test_noalloc_forward_matches_workspace_forward_twice(b, s):
    # For M > 64 both entry points run the same tile kernels, which are deterministic:
    # the results must be the same bits, on each of two calls in a row.
    for call, seed in enumerate((21, 22)):      # two calls in a row, different inputs
        _, x, W1, W2, _ = workloads.make_block(s, seed=seed)
        x, W1, W2 = x.cuda(), W1.cuda(), W2.cuda()
        pre_ref, y_ref = b.swiglu_mlp_fwd(x, W1, W2)
        pre, y = _noalloc_via_abi(b, x, W1, W2)
        assert b.swiglu_mlp_device_status() == 0
        assert torch.equal(pre, pre_ref), f"preact (call {call})"
        assert torch.equal(y, y_ref), f"y (call {call})"


@pytest.mark.parametrize("s", [Shape(16, 128, 384, 512), Shape(64, 256, 520, 136)],
                         ids=lambda s: f"M{s.M}_D{s.D}_H{s.H}_Do{s.Dout}")
def test_noalloc_few_tokens_against_oracle_twice(b, s):
    # For M <= 64 the ordinary forward takes the few-token kernels while the
    # allocation-free one keeps the tile kernels: the two are compared through the
    # oracle (and with each other within the same bar), on two calls in a row.
    import oracle
    for call, seed in enumerate((23, 24)):
        _, x, W1, W2, _ = workloads.make_block(s, seed=seed, gate_sweep=True)
        p_ref, _, y_ref = oracle.fwd(x, W1, W2)
        xd, W1d, W2d = x.cuda(), W1.cuda(), W2.cuda()
        pre, y = _noalloc_via_abi(b, xd, W1d, W2d)
        pre_ws, y_ws = b.swiglu_mlp_fwd(xd, W1d, W2d)
        assert b.swiglu_mlp_device_status() == 0
        parity(pre, p_ref, f"preact (call {call})")
        parity(y, y_ref, f"y (call {call})")
        parity(pre, pre_ws.float().cpu().double().numpy(), f"preact vs swiglu_mlp_fwd (call {call})")
        parity(y, y_ws.float().cpu().double().numpy(), f"y vs swiglu_mlp_fwd (call {call})")


def test_noalloc_rejects_sizes_beyond_the_builtin_scratch(b):
    # M*H*2 bytes one element over 64 MiB: refused before any work is enqueued
    A16 = ctypes.c_void_p(0x10000)
    H = 8192
    M = (64 * 1024 * 1024) // (2 * H) + 1
    st = b.lib().swiglu_mlp_fwd_noalloc(A16, A16, A16, A16, A16, M, 64, H, 64, None)
    assert st == 4                                   # SWIGLU_ERR_WORKSPACE_TOO_SMALL
    assert b"built-in scratch" in b.lib().swiglu_mlp_last_error_detail()
