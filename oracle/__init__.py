"""CPU oracle for the SwiGLU MLP block -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never uses it and it
never uses the CUDA library: the two share no code.  Inputs are bf16 bit
patterns (``uint16`` numpy arrays or ``torch.bfloat16`` CPU tensors) or, for
the finite-difference pins, fp64 arrays; every result is an fp64 numpy array.

The arithmetic lives in ``swiglu_oracle.c`` (plain C loops, fp64, OpenMP over
independent outputs); this module only compiles it on demand and marshals
arguments.  Formulas and rounding points are documented there; they follow the
"SwiGLU MLP Drop-H technical report" (lgystoic.github.io/notes/
swiglu-mlp-drop-h/), forward/backward formulas and fused-kernel pseudo-code,
and the "SwiGLU MLP forward/backward optimization" note (lgystoic.github.io/
notes/swiglu-mlp-forward-backward-optimization/), section 2 (silu' forms).

Parity pins (tests/test_oracle.py): silu' against a central finite difference;
the whole gradient chain against finite differences of L = sum(dy * y); the
unrounded chain against torch fp64 autograd; bf16 rounding against torch's
fp32->bf16 conversion and hand-worked ties; closed forms at g = 0, +-20;
permutation weights, where every product reduces to a gather; for the
mixture-of-experts functions, experts built as hidden-unit permutations and
power-of-two scalings of one dense block, whose outputs are then known
transforms of the dense block's; for the FP8 forward, E4M3 decoding against
torch's float8_e4m3fn, encoding against torch's rounding, hand-worked ties and
saturation, and the FP8 forward against the bf16 oracle on the dequantised
inputs and an fp64 matmul of the dequantised codes.  No function here is
"parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "swiglu_oracle.c")
_LIB = os.path.join(_HERE, "libswiglu_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, no fast-math, OpenMP) if stale."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
               "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            d, i64, i32 = ctypes.c_double, ctypes.c_int64, ctypes.c_int
            vp = ctypes.c_void_p
            lib.oracle_round_bf16.restype = d
            lib.oracle_round_bf16.argtypes = [d]
            for f in ("oracle_sigmoid", "oracle_silu", "oracle_silu_prime"):
                getattr(lib, f).restype = d
                getattr(lib, f).argtypes = [d]
            lib.oracle_swiglu_fwd.restype = i32
            lib.oracle_swiglu_fwd.argtypes = [vp, vp, vp, i32, i64, i64, i64, i64, vp, i64, i32, i32,
                                              vp, vp, vp]
            lib.oracle_swiglu_bwd_rows.restype = i32
            lib.oracle_swiglu_bwd_rows.argtypes = [vp, vp, vp, vp, i32, i64, i64, i64, i64, vp, i64,
                                                   i32, i32, vp, vp, vp, vp]
            lib.oracle_swiglu_bwd_cols.restype = i32
            lib.oracle_swiglu_bwd_cols.argtypes = [vp, vp, vp, vp, i32, i64, i64, i64, i64, vp, i64,
                                                   i32, vp, vp]
            lib.oracle_num_threads.restype = i32
            lib.oracle_num_threads.argtypes = []
            lib.oracle_e4m3_decode.restype = d
            lib.oracle_e4m3_decode.argtypes = [i32]
            lib.oracle_e4m3_encode.restype = i32
            lib.oracle_e4m3_encode.argtypes = [d]
            lib.oracle_swiglu_fwd_fp8.restype = i32
            lib.oracle_swiglu_fwd_fp8.argtypes = [vp, vp, vp, d, d, d, d, i64, i64, i64, i64, vp, i64,
                                                  vp, vp, vp, vp]
            _lib = lib
    return _lib


def _bits(a) -> np.ndarray:
    """bf16 tensor / uint16 bit-pattern array / float64 array -> contiguous numpy array."""
    if hasattr(a, "dtype") and str(a.dtype) == "torch.bfloat16":
        import torch
        return a.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    if hasattr(a, "dtype") and str(a.dtype) == "torch.float64":
        return a.detach().cpu().contiguous().numpy()
    arr = np.ascontiguousarray(a)
    if arr.dtype not in (np.uint16, np.float64):
        raise TypeError(f"expected bf16 bit patterns (uint16) or float64, got {arr.dtype}")
    return arr


def _kind(*arrs) -> int:
    """0 when every input is bf16 bits, 1 when every input is fp64."""
    kinds = {a.dtype for a in arrs}
    if len(kinds) != 1:
        raise TypeError("inputs must be all bf16 or all float64")
    return int(kinds.pop() == np.float64)


def _index(idx, n):
    if idx is None:
        return None, n
    arr = np.ascontiguousarray(np.asarray(idx, dtype=np.int64))
    return arr, arr.size


def _ptr(a):
    return None if a is None else a.ctypes.data


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def round_bf16(v: float) -> float:
    return float(_load().oracle_round_bf16(float(v)))


def sigmoid(g: float) -> float:
    return float(_load().oracle_sigmoid(float(g)))


def silu(g: float) -> float:
    return float(_load().oracle_silu(float(g)))


def silu_prime(g: float) -> float:
    return float(_load().oracle_silu_prime(float(g)))


def fwd(x, W1, W2, rows=None, round_intermediates: bool = True, residual: bool = False):
    """Forward for the selected token rows (all rows when ``rows`` is None).
    ``residual``: the residual block y = x + MLP(x) (D == Dout).

    Returns (preact [n,2H], h [n,H], y [n,Dout]) as fp64 arrays.
    """
    xb, w1b, w2b = _bits(x), _bits(W1), _bits(W2)
    M, D = xb.shape
    H = w1b.shape[0] // 2
    Dout = w2b.shape[0]
    if w1b.shape != (2 * H, D) or w2b.shape != (Dout, H) or (residual and D != Dout):
        raise ValueError("shape mismatch")
    ridx, n = _index(rows, M)
    preact = np.empty((n, 2 * H))
    h = np.empty((n, H))
    y = np.empty((n, Dout))
    rc = _load().oracle_swiglu_fwd(_ptr(xb), _ptr(w1b), _ptr(w2b), _kind(xb, w1b, w2b),
                                   M, D, H, Dout, _ptr(ridx), n,
                                   int(round_intermediates), int(residual), _ptr(preact), _ptr(h), _ptr(y))
    if rc != 0:
        raise MemoryError("oracle_swiglu_fwd failed")
    return preact, h, y


def bwd_rows(W1, W2, preact, dy, rows=None, round_intermediates: bool = True, residual: bool = False):
    """Row-wise backward outputs for the selected token rows (``residual``: dx += dy).

    Returns (grad_h [n,H], grad_preact [n,2H], h [n,H], dx [n,D]) as fp64 arrays.
    """
    w1b, w2b, pb, dyb = _bits(W1), _bits(W2), _bits(preact), _bits(dy)
    H2, D = w1b.shape
    H = H2 // 2
    Dout = w2b.shape[0]
    M = pb.shape[0]
    if pb.shape != (M, 2 * H) or dyb.shape != (M, Dout) or w2b.shape != (Dout, H) or (residual and D != Dout):
        raise ValueError("shape mismatch")
    ridx, n = _index(rows, M)
    gh = np.empty((n, H))
    gp = np.empty((n, 2 * H))
    h = np.empty((n, H))
    dx = np.empty((n, D))
    rc = _load().oracle_swiglu_bwd_rows(_ptr(w1b), _ptr(w2b), _ptr(pb), _ptr(dyb),
                                        _kind(w1b, w2b, pb, dyb), M, D, H, Dout,
                                        _ptr(ridx), n, int(round_intermediates), int(residual),
                                        _ptr(gh), _ptr(gp), _ptr(h), _ptr(dx))
    if rc != 0:
        raise MemoryError("oracle_swiglu_bwd_rows failed")
    return gh, gp, h, dx


def bwd_cols(x, W2, preact, dy, cols=None, round_intermediates: bool = True):
    """Weight gradients for the selected hidden indices j (all j when ``cols`` is None).

    Returns (dW2_cols [n,Dout] -- row k is the column dW2[:, cols[k]],
             dW1_left [n,D]    -- row k is dW1[cols[k], :],
             dW1_gate [n,D]    -- row k is dW1[H + cols[k], :]).
    """
    xb, w2b, pb, dyb = _bits(x), _bits(W2), _bits(preact), _bits(dy)
    M, D = xb.shape
    Dout, H = w2b.shape
    if pb.shape != (M, 2 * H) or dyb.shape != (M, Dout):
        raise ValueError("shape mismatch")
    cidx, n = _index(cols, H)
    dW2c = np.empty((n, Dout))
    dW1 = np.empty((2 * n, D))
    rc = _load().oracle_swiglu_bwd_cols(_ptr(xb), _ptr(w2b), _ptr(pb), _ptr(dyb),
                                        _kind(xb, w2b, pb, dyb), M, D, H, Dout,
                                        _ptr(cidx), n, int(round_intermediates),
                                        _ptr(dW2c), _ptr(dW1))
    if rc != 0:
        raise MemoryError("oracle_swiglu_bwd_cols failed")
    return dW2c, dW1[:n], dW1[n:]


def bwd_full(x, W1, W2, preact, dy, round_intermediates: bool = True, residual: bool = False):
    """Whole backward on a small problem: (grad_h, grad_preact, h, dx, dW1 [2H,D], dW2 [Dout,H])."""
    gh, gp, h, dx = bwd_rows(W1, W2, preact, dy, None, round_intermediates, residual)
    dW2c, dW1l, dW1g = bwd_cols(x, W2, preact, dy, None, round_intermediates)
    return gh, gp, h, dx, np.concatenate([dW1l, dW1g], axis=0), dW2c.T.copy()


# ---------------------------------------------------------------------------- mixture of experts
#
# "Lesson 24: MLP, GEMM and operator fusion in the Transformer" (lincklin.cn), section 41
# (each expert of an MoE layer is an MLP of its own; every token is routed to one
# expert) and section 42 (the experts' GEMMs differ only in their row counts M_e).
# Layout: the tokens arrive grouped by expert -- expert e owns rows
# [off_e, off_e + counts[e]) of x, dy, preact, y and dx, with off_e the sum of the
# counts before it -- and the weights are stacked per expert: W1 [E, 2H, D],
# W2 [E, Dout, H].  Each expert's rows go through the block above with that
# expert's weights; nothing else is computed.

def expert_offsets(counts) -> np.ndarray:
    """[E + 1] row offsets of the experts' segments."""
    c = np.asarray(counts, dtype=np.int64)
    if c.ndim != 1 or (c < 0).any():
        raise ValueError("counts must be a 1-D array of non-negative ints")
    return np.concatenate([[0], np.cumsum(c)])


def _moe_shapes(W1, W2, counts):
    w1b, w2b = _bits(W1), _bits(W2)
    E, H2, D = w1b.shape
    Dout, H = w2b.shape[1], w2b.shape[2]
    off = expert_offsets(counts)
    if w2b.shape[0] != E or H2 != 2 * H or off.size != E + 1:
        raise ValueError("shape mismatch")
    return w1b, w2b, off, E, D, H, Dout


def moe_fwd(x, W1, W2, counts, round_intermediates: bool = True):
    """Forward of every expert on its rows: (preact [T,2H], h [T,H], y [T,Dout])."""
    xb = _bits(x)
    w1b, w2b, off, E, D, H, Dout = _moe_shapes(W1, W2, counts)
    T = xb.shape[0]
    if off[-1] != T:
        raise ValueError("counts do not sum to the number of rows")
    preact, h, y = np.zeros((T, 2 * H)), np.zeros((T, H)), np.zeros((T, Dout))
    for e in range(E):
        a, b = off[e], off[e + 1]
        if b > a:
            preact[a:b], h[a:b], y[a:b] = fwd(xb[a:b], w1b[e], w2b[e], None, round_intermediates)
    return preact, h, y


def moe_bwd_full(x, W1, W2, preact, dy, counts, round_intermediates: bool = True):
    """Backward of every expert on its rows:
    (grad_h [T,H], grad_preact [T,2H], h [T,H], dx [T,D], dW1 [E,2H,D], dW2 [E,Dout,H]).
    An expert that received no rows has zero weight gradients."""
    xb, pb, dyb = _bits(x), _bits(preact), _bits(dy)
    w1b, w2b, off, E, D, H, Dout = _moe_shapes(W1, W2, counts)
    T = xb.shape[0]
    if off[-1] != T:
        raise ValueError("counts do not sum to the number of rows")
    gh, gp, h, dx = np.zeros((T, H)), np.zeros((T, 2 * H)), np.zeros((T, H)), np.zeros((T, D))
    dW1, dW2 = np.zeros((E, 2 * H, D)), np.zeros((E, Dout, H))
    for e in range(E):
        a, b = off[e], off[e + 1]
        if b > a:
            gh[a:b], gp[a:b], h[a:b], dx[a:b], dW1[e], dW2[e] = bwd_full(
                xb[a:b], w1b[e], w2b[e], pb[a:b], dyb[a:b], round_intermediates)
    return gh, gp, h, dx, dW1, dW2


def moe_rows(x, W1, W2, preact, dy, counts, rows):
    """Sampled token rows (global indices): (preact, y, grad_preact, h, dx) of those rows,
    each computed by its own expert."""
    xb, pb, dyb = _bits(x), _bits(preact), _bits(dy)
    w1b, w2b, off, E, D, H, Dout = _moe_shapes(W1, W2, counts)
    rows = np.asarray(rows, dtype=np.int64)
    out = [np.zeros((rows.size, n)) for n in (2 * H, Dout, 2 * H, H, D)]
    for k, r in enumerate(rows):
        e = int(np.searchsorted(off, r, side="right") - 1)
        local = [r - off[e]]
        seg = slice(off[e], off[e + 1])
        p, _, yv = fwd(xb[seg], w1b[e], w2b[e], rows=local)
        _, gpv, hv, dxv = bwd_rows(w1b[e], w2b[e], pb[seg], dyb[seg], rows=local)
        for o, v in zip(out, (p, yv, gpv, hv, dxv)):
            o[k] = v[0]
    return tuple(out)


def moe_cols(x, W2, preact, dy, counts, expert, cols):
    """Expert `expert`'s weight gradients for the selected hidden indices, as bwd_cols."""
    xb, pb, dyb = _bits(x), _bits(preact), _bits(dy)
    w2b = _bits(W2)
    off = expert_offsets(counts)
    a, b = off[expert], off[expert + 1]
    Dout, H = w2b.shape[1], w2b.shape[2]
    n = len(cols)
    if b == a:
        return np.zeros((n, Dout)), np.zeros((n, xb.shape[1])), np.zeros((n, xb.shape[1]))
    return bwd_cols(xb[a:b], w2b[expert], pb[a:b], dyb[a:b], cols=cols)


# ---------------------------------------------------------------------------- FP8 forward
#
# "Lesson 24: MLP, GEMM and operator fusion in the Transformer" (lincklin.cn),
# section 26 (the quantised GEMM epilogue, y = sat8(round(s * acc + b))) and
# section 31 (8-bit weights for the weight-bound decode).  Formats and rounding
# points are documented in swiglu_oracle.c.

def e4m3_decode(code: int) -> float:
    """Value of an FP8 E4M3 code (NaN for the NaN codes)."""
    return float(_load().oracle_e4m3_decode(int(code)))


def e4m3_encode(v: float) -> int:
    """Nearest E4M3 code, ties to even, saturating at +-448."""
    return int(_load().oracle_e4m3_encode(float(v)))


def _codes(a) -> np.ndarray:
    """torch float8_e4m3fn / uint8 tensor or uint8 array -> contiguous uint8 codes."""
    if hasattr(a, "dtype") and str(a.dtype) in ("torch.float8_e4m3fn", "torch.uint8"):
        import torch
        return a.detach().cpu().contiguous().view(torch.uint8).numpy()
    arr = np.ascontiguousarray(a)
    if arr.dtype != np.uint8:
        raise TypeError(f"expected E4M3 codes (uint8), got {arr.dtype}")
    return arr


def fwd_fp8(x8, W1_8, W2_8, s_x: float, s_w1: float, s_w2: float, s_h: float, rows=None):
    """FP8 forward for the selected token rows (all rows when ``rows`` is None).

    Returns (preact [n,2H] bf16-rounded, h [n,H] before quantisation, h8 [n,H] E4M3
    codes (uint8), y [n,Dout] unrounded), fp64 except h8.
    """
    xb, w1b, w2b = _codes(x8), _codes(W1_8), _codes(W2_8)
    M, D = xb.shape
    H = w1b.shape[0] // 2
    Dout = w2b.shape[0]
    if w1b.shape != (2 * H, D) or w2b.shape != (Dout, H):
        raise ValueError("shape mismatch")
    ridx, n = _index(rows, M)
    preact = np.empty((n, 2 * H))
    hpre = np.empty((n, H))
    h8 = np.empty((n, H), dtype=np.uint8)
    y = np.empty((n, Dout))
    rc = _load().oracle_swiglu_fwd_fp8(_ptr(xb), _ptr(w1b), _ptr(w2b), float(s_x), float(s_w1), float(s_w2),
                                       float(s_h), M, D, H, Dout, _ptr(ridx), n,
                                       _ptr(preact), _ptr(hpre), _ptr(h8), _ptr(y))
    if rc != 0:
        raise MemoryError("oracle_swiglu_fwd_fp8 failed")
    return preact, hpre, h8, y
