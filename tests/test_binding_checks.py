"""The Python binding checks every tensor before anything reaches the library (CPU only).

The kernels address their operands through tensor maps built from the sizes, so a
buffer of the wrong shape, dtype or device would be read or written past its end.
The binding derives the sizes from x and the weights and checks every other tensor,
inputs and caller-supplied outputs, against them.  On CPU tensors a call that passes
every check stops at the last one, "must live on a CUDA device": the calls below
are the ones the library's own users make (tests, bench, stack, pipeline, smoke).
"""
import pytest
import torch

from helpers import ensure_library

CUDA = "must live on a CUDA device"
bf, f8, u8 = torch.bfloat16, torch.float8_e4m3fn, torch.uint8
M, D, H, Do = 48, 32, 64, 40


@pytest.fixture(scope="module")
def b():
    ensure_library()
    from bwd_gemm_epilogue_gb300 import binding
    binding.lib()
    return binding


def z(*shape, dtype=bf, device="cpu"):
    return torch.zeros(*shape, dtype=dtype, device=device)


def legal_calls(b):
    x, W1, W2 = z(M, D), z(2 * H, D), z(Do, H)
    pre, dy = z(M, 2 * H), z(M, Do)
    xs, W1s, W2s = z(M, D), z(2 * H, D), z(D, H)                 # D == Dout: residual, stack
    E, counts = 3, [20, 0, 28]
    W1e, W2e = z(E, 2 * H, D), z(E, Do, H)
    ws = torch.zeros(16, dtype=u8)
    x8, W18, W28 = z(M, D, dtype=f8), z(2 * H, D, dtype=f8), z(Do, H, dtype=f8)
    sc = dict(s_x=1.0, s_w1=1.0, s_w2=1.0, s_h=1.0)
    calls = {
        "fwd": lambda: b.swiglu_mlp_fwd(x, W1, W2),
        "fwd, caller buffers": lambda: b.swiglu_mlp_fwd(x, W1, W2, z(M, 2 * H), z(M, Do), ws),
        "fwd residual": lambda: b.swiglu_mlp_fwd(xs, W1s, W2s, residual=True),
        "fwd noalloc": lambda: b.swiglu_mlp_fwd_noalloc(x, W1, W2),
        "bwd": lambda: b.swiglu_mlp_bwd(x, W1, W2, pre, dy),
        "bwd, caller buffers": lambda: b.swiglu_mlp_bwd(x, W1, W2, pre, dy, z(M, D), z(2 * H, D), z(Do, H), ws),
        "bwd residual": lambda: b.swiglu_mlp_bwd(xs, W1s, W2s, pre, z(M, D), residual=True),
        "bwd empty batch": lambda: b.swiglu_mlp_bwd(z(0, D), W1, W2, z(0, 2 * H), z(0, Do),
                                                    dW1=z(2 * H, D), dW2=z(Do, H)),
        "fused": lambda: b.swiglu_mlp_fused_grad_preact(dy, W2, pre),
        "fused, caller buffers": lambda: b.swiglu_mlp_fused_grad_preact(dy, W2, pre, z(M, 2 * H), z(M, H)),
        "fp8": lambda: b.swiglu_mlp_fwd_fp8(x8, W18, W28, **sc),
        "fp8, h8 and y only": lambda: b.swiglu_mlp_fwd_fp8(x8, W18, W28, h8=z(M, H, dtype=f8), y=z(M, Do),
                                                           store_preact=False, **sc),
        "moe fwd": lambda: b.swiglu_moe_fwd(x, W1e, W2e, counts),
        "moe fwd, caller buffers": lambda: b.swiglu_moe_fwd(x, W1e, W2e, counts, z(M, 2 * H), z(M, Do), ws),
        "moe bwd": lambda: b.swiglu_moe_bwd(x, W1e, W2e, pre, dy, counts),
        "moe bwd, caller buffers": lambda: b.swiglu_moe_bwd(x, W1e, W2e, pre, dy, counts, z(M, D),
                                                            z(E, 2 * H, D), z(E, Do, H), ws),
        "moe empty": lambda: b.swiglu_moe_bwd(z(0, D), W1e, W2e, z(0, 2 * H), z(0, Do), [0, 0, 0],
                                              dW1=z(E, 2 * H, D), dW2=z(E, Do, H)),
    }
    for a_mn in (False, True):
        for b_mn in (False, True):
            A = z(D, M) if a_mn else z(M, D)                       # C [M, Do] = A B^T, K = D
            B = z(D, Do) if b_mn else z(Do, D)
            calls[f"gemm a_mn={a_mn} b_mn={b_mn}"] = (
                lambda A=A, B=B, a=a_mn, c=b_mn: b.swiglu_mlp_gemm_bf16(A, B, M, Do, D, a, c))
    calls["gemm, caller C"] = lambda: b.swiglu_mlp_gemm_bf16(z(M, D), z(Do, D), M, Do, D, False, False, z(M, Do))
    return calls


def test_the_library_users_calls_pass_every_check(b):
    for name, call in legal_calls(b).items():
        with pytest.raises(ValueError, match=CUDA):
            call()


def _wrong_calls(b):
    x, W1, W2 = z(M, D), z(2 * H, D), z(Do, H)
    pre, dy = z(M, 2 * H), z(M, Do)
    W1e, W2e = z(3, 2 * H, D), z(3, Do, H)
    x8, W18, W28 = z(M, D, dtype=f8), z(2 * H, D, dtype=f8), z(Do, H, dtype=f8)
    sc = dict(s_x=1.0, s_w1=1.0, s_w2=1.0, s_h=1.0)
    return [
        (lambda: b.swiglu_mlp_fwd(x, W1, W2, preact=z(M, H)), ValueError, "preact: shape"),
        (lambda: b.swiglu_mlp_fwd(x, W1, W2, y=z(M, Do, dtype=torch.float32)), TypeError, "y: torch.float32"),
        (lambda: b.swiglu_mlp_fwd(x.float(), W1, W2), TypeError, "x: torch.float32"),
        (lambda: b.swiglu_mlp_fwd(x, W1, W2, y=z(M, Do, device="meta")), ValueError, "y: on meta"),
        (lambda: b.swiglu_mlp_fwd(x, W1, W2, workspace=z(16, dtype=u8, device="meta")), ValueError,
         "workspace: on meta"),
        (lambda: b.swiglu_mlp_fwd_noalloc(x, W1, W2, y=z(M + 1, Do)), ValueError, "y: shape"),
        (lambda: b.swiglu_mlp_bwd(x, W1, W2, pre, z(M, D)), ValueError, "dy: shape"),
        (lambda: b.swiglu_mlp_bwd(x, W1, W2, z(M, 2 * H - 8), dy), ValueError, "preact: shape"),
        (lambda: b.swiglu_mlp_bwd(x, W1, W2, pre, dy, dW2=z(H, Do)), ValueError, "dW2: shape"),
        (lambda: b.swiglu_mlp_bwd(x, W1, W2, pre, dy, dx=z(M, D, dtype=u8)), TypeError, "dx: torch.uint8"),
        (lambda: b.swiglu_mlp_fused_grad_preact(dy, W2, pre, h=z(M, 2 * H)), ValueError, "h: shape"),
        (lambda: b.swiglu_mlp_fused_grad_preact(dy.float(), W2, pre), TypeError, "dy: torch.float32"),
        (lambda: b.swiglu_mlp_fwd_fp8(x, W1, W2, **sc), TypeError, "x: torch.bfloat16"),
        (lambda: b.swiglu_mlp_fwd_fp8(x8, W18, W28, h8=z(M, H), **sc), TypeError, "h8: torch.bfloat16"),
        (lambda: b.swiglu_mlp_gemm_bf16(z(M, D), z(Do, D), M, Do, D, True, False), ValueError, "A: shape"),
        (lambda: b.swiglu_mlp_gemm_bf16(z(M, D), z(Do, D), M, Do, D, False, True), ValueError, "B: shape"),
        (lambda: b.swiglu_mlp_gemm_bf16(z(M, D), z(Do, D), M, Do, D, False, False, z(Do, M)), ValueError,
         "C: shape"),
        (lambda: b.swiglu_moe_fwd(x, W1e, W2e, [20, 0, 28], y=z(M, D)), ValueError, "y: shape"),
        (lambda: b.swiglu_moe_bwd(x, W1e, W2e, z(M, H), dy, [20, 0, 28]), ValueError, "preact: shape"),
        (lambda: b.swiglu_moe_bwd(x, W1e, W2e, pre, dy, [20, 0, 28], dW1=z(2 * H, D)), ValueError, "dW1: shape"),
        (lambda: b.swiglu_moe_fwd(x, W1e.float(), W2e, [20, 0, 28]), TypeError, "W1: torch.float32"),
    ]


def test_wrong_buffers_are_refused_by_name(b):
    for call, err, match in _wrong_calls(b):
        with pytest.raises(err, match=match):
            call()


def test_tensors_on_another_device_than_the_current_one_are_refused(b, monkeypatch):
    # The library launches on the current CUDA device; tensors on another GPU would be
    # addressed from the wrong one.  The binding refuses before any launch.
    monkeypatch.setattr(torch.cuda, "current_device", lambda: 1)
    with pytest.raises(ValueError, match="current CUDA device"):
        b._stream(torch.device("cuda", 0))
