"""Host-side checks of the C ABI: the library loads, exports every symbol the
header declares, and rejects bad arguments before touching the GPU."""
import ctypes

import pytest

from helpers import ensure_library, header_functions


@pytest.fixture(scope="module")
def lib():
    ensure_library()
    from bwd_gemm_epilogue_gb300 import binding
    return binding.lib()


def test_library_exports_every_declared_symbol(lib):
    from bwd_gemm_epilogue_gb300 import binding
    names = header_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
        assert n in binding.SIGNATURES, f"binding misses {n}"


def test_workspace_sizes():
    from bwd_gemm_epilogue_gb300 import binding as b
    M, D, H, Dout = 11136, 3584, 14336, 3584
    # h, then the down projection's split-tile counters and fp32 sums
    assert b.swiglu_mlp_fwd_workspace_size(M, D, H, Dout) == M * H * 2 + 20480 + 80 * 524288
    assert b.swiglu_mlp_bwd_workspace_size(M, D, H, Dout) == M * H * 2 + M * 2 * H * 2
    assert b.swiglu_mlp_fwd_workspace_size(0, D, H, Dout) == 0
    # ragged: each buffer starts on a 256-byte boundary
    assert b.swiglu_mlp_bwd_workspace_size(3, 8, 8, 8) == 256 + 256 + 512 + 512   # + small-M fp32 sums
    assert b.swiglu_mlp_bwd_workspace_size(65, 8, 8, 8) == 1280 + 2304            # M > 64: h, grad_preact
    # small-M forward: h, then one fp32 partial plane per K split of preact^T [2H, 16] and of
    # y^T [Dout, 16]; for 16 tokens at 4096 x 11008 the split-K plan (152 SMs) uses 7 and 14
    assert b.swiglu_mlp_fwd_workspace_size(16, 4096, 11008, 4096) == \
        16 * 11008 * 2 + 7 * 2 * 11008 * 16 * 4 + 14 * 4096 * 16 * 4


def test_strerror_and_version():
    from bwd_gemm_epilogue_gb300 import binding as b
    for code, name in b.STATUS_NAMES.items():
        assert b.swiglu_mlp_strerror(code).startswith(name)
    assert b.swiglu_mlp_abi_version() == 201


A16 = 0x10000          # fake, 16-byte aligned "device" addresses: validation never dereferences them
BIG = 1 << 40


def _fwd(lib, x=A16, w1=A16, w2=A16, pre=A16, y=A16, M=128, D=256, H=512, Do=256, ws=A16, wsb=BIG):
    return lib.swiglu_mlp_fwd(x, w1, w2, pre, y, M, D, H, Do, ws, wsb, None)


def _bwd(lib, ptr=A16, M=128, D=256, H=512, Do=256, ws=A16, wsb=BIG, **over):
    p = dict(x=ptr, w1=ptr, w2=ptr, pre=ptr, dy=ptr, dx=ptr, dw1=ptr, dw2=ptr)
    p.update(over)
    return lib.swiglu_mlp_bwd(p["x"], p["w1"], p["w2"], p["pre"], p["dy"], p["dx"], p["dw1"], p["dw2"],
                              M, D, H, Do, ws, wsb, None)


def test_argument_validation_before_launch(lib):
    INVALID, SHAPE, MISALIGNED, WS = 1, 2, 3, 4
    assert _fwd(lib, D=100) == SHAPE                 # not a multiple of 8
    assert _fwd(lib, H=0) == INVALID
    assert _fwd(lib, Do=-8) == INVALID
    assert _fwd(lib, M=-1) == INVALID
    assert _fwd(lib, M=1 << 31) == SHAPE
    assert _fwd(lib, x=None) == INVALID
    assert _fwd(lib, y=A16 + 8) == MISALIGNED
    assert _fwd(lib, wsb=128 * 512 * 2 - 1) == WS
    assert _fwd(lib, M=0) == 0                       # empty input: nothing to do
    assert _bwd(lib, H=12) == SHAPE
    assert _bwd(lib, dw1=None) == INVALID
    assert _bwd(lib, pre=A16 + 2) == MISALIGNED
    assert _bwd(lib, wsb=100) == WS
    assert lib.swiglu_mlp_fused_grad_preact(A16, A16, A16, A16, None, 4, 8, 8, None) == INVALID
    assert lib.swiglu_mlp_fused_grad_preact(A16, A16, A16, A16, A16, 4, 8, 9, None) == SHAPE
    assert lib.swiglu_mlp_fused_grad_preact(A16, A16, A16, A16, A16, 0, 8, 8, None) == 0
    assert lib.swiglu_mlp_gemm_bf16(A16, A16, A16, 0, 8, 8, 0, 0, None) == INVALID
    assert lib.swiglu_mlp_gemm_bf16(A16, A16, A16, 5, 8, 12, 0, 0, None) == SHAPE   # K-major A needs K % 8
    assert lib.swiglu_mlp_gemm_bf16(A16, A16, A16, 5, 8, 12, 1, 1, None) == SHAPE   # MN-major A needs M % 8
    assert lib.swiglu_mlp_gemm_bf16(A16 + 4, A16, A16, 8, 8, 8, 0, 0, None) == MISALIGNED


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    from bwd_gemm_epilogue_gb300 import binding as b
    monkeypatch.setattr(b, "_lib", None)
    monkeypatch.setattr(b, "LIB_PATH", str(tmp_path / "nope.so"))
    with pytest.raises(RuntimeError, match="build the CUDA library"):
        b.lib()


# ---------------------------------------------------------------------------- mixture of experts

def _counts(vals):
    arr = (ctypes.c_int64 * len(vals))(*vals)
    return ctypes.cast(arr, ctypes.c_void_p), arr


def test_moe_workspace_sizes(lib):
    c, keep = _counts([32, 120, 8, 64])
    T, H = 224, 512
    fwd = lib.swiglu_moe_fwd_workspace_size(c, 4, 256, H, 256)
    bwd = lib.swiglu_moe_bwd_workspace_size(c, 4, 256, H, 256)
    assert fwd >= T * H * 2 and bwd >= T * H * 2 + T * 2 * H * 2
    c2, keep2 = _counts([32, 120, 8, 6400])
    assert lib.swiglu_moe_fwd_workspace_size(c2, 4, 256, H, 256) > fwd      # more rows, more tiles
    bad, keep3 = _counts([3, -1])
    assert lib.swiglu_moe_fwd_workspace_size(bad, 2, 256, H, 256) == 0
    assert lib.swiglu_moe_bwd_workspace_size(None, 2, 256, H, 256) == 0
    assert lib.swiglu_moe_fwd_workspace_size(c, 0, 256, H, 256) == 0


def test_moe_argument_errors(lib):
    c, keep = _counts([32, 120, 8, 64])

    def fwd(x=A16, ws=A16, wsb=BIG, D=256, H=512, Do=256, counts=c, E=4):
        return lib.swiglu_moe_fwd(x, A16, A16, A16, A16, counts, E, D, H, Do, ws, wsb, None)

    assert fwd(x=A16 + 8) == 3                 # misaligned
    assert fwd(x=None) == 1                    # null input
    assert fwd(D=100) == 2                     # D not a multiple of 8
    assert fwd(wsb=64) == 4                    # workspace too small
    assert fwd(counts=None) == 1
    assert fwd(E=683) == 1                     # more experts than one launch's table indexes
    big, keep2 = _counts([1 << 30, 1 << 30])
    assert fwd(counts=big, E=2) == 1           # T >= 2^31
    assert lib.swiglu_moe_bwd(A16, A16, A16, A16, A16, A16, A16, A16 + 4, c, 4, 256, 512, 256,
                              A16, BIG, None) == 3


def test_fp8_forward_argument_errors(lib):
    def f(D=256, H=512, Do=256, sh=1.0, x=A16, h8=A16):
        return lib.swiglu_mlp_fwd_fp8(x, A16, A16, 1.0, 1.0, 1.0, sh, None, h8, A16, 128, D, H, Do, None, 0, None)

    assert f(D=264) == 2                       # D not a multiple of 16
    assert f(H=520) == 2                       # H not a multiple of 16
    assert f(sh=0.0) == 1 and f(sh=-1.0) == 1  # scales must be positive
    assert f(x=None) == 1
    assert f(h8=A16 + 8) == 3
    # few tokens need fp32 workspace sums
    # fp32 partial planes: 7 K splits of preact^T, 13 of y^T (128-value FP8 k-blocks)
    assert lib.swiglu_mlp_fwd_fp8_workspace_size(16, 4096, 11008, 4096) == 7 * 2 * 11008 * 16 * 4 + 13 * 4096 * 16 * 4
    assert lib.swiglu_mlp_fwd_fp8_workspace_size(65, 4096, 11008, 4096) == 0
    assert lib.swiglu_mlp_fwd_fp8(A16, A16, A16, 1.0, 1.0, 1.0, 1.0, None, A16, A16, 16, 256, 512, 256,
                                  None, 0, None) == 4
