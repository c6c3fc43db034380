"""FLOP and byte ledger of the SwiGLU MLP block's kernels.

FLOPs count 2 per multiply-add.  The backward's four GEMMs come in the ratio
grad_h : dW2 : dx : dW1 = 1 : 1 : 2 : 2, which makes the backward exactly twice
the forward -- the ledger of the "SwiGLU MLP forward/backward optimization"
note (section 3, 116 + 116 + 232 + 232 = 696 GF = 2 x 348 GF).

Bytes are the compulsory HBM traffic of each kernel: every operand read once,
every output written once, all bf16 (2 bytes per element).
"""
from __future__ import annotations

BF16 = 2


def gemm_flops(M: int, D: int, H: int, Dout: int) -> dict:
    f = {
        "fwd_preact": 2 * M * D * 2 * H,   # x @ W1^T, SwiGLU epilogue
        "fwd_down": 2 * M * H * Dout,      # h @ W2^T
        "bwd_grad_h": 2 * M * Dout * H,    # dy @ W2, SwiGLU-backward epilogue
        "bwd_dW2": 2 * Dout * M * H,       # dy^T @ h
        "bwd_dx": 2 * M * 2 * H * D,       # grad_preact @ W1
        "bwd_dW1": 2 * 2 * H * M * D,      # grad_preact^T @ x, one merged product
    }
    f["bwd_gemms"] = f["bwd_dW2"] + f["bwd_dx"] + f["bwd_dW1"]   # the grouped launch
    f["fwd"] = f["fwd_preact"] + f["fwd_down"]
    f["bwd"] = f["bwd_grad_h"] + f["bwd_dW2"] + f["bwd_dx"] + f["bwd_dW1"]
    f["step"] = f["fwd"] + f["bwd"]
    return f


def kernel_bytes(M: int, D: int, H: int, Dout: int, experts: int = 1) -> dict:
    """Compulsory HBM bytes per launch of each kernel.  `experts`: the number of
    weight sets read (and weight gradients written) -- the experts that received
    rows, for a mixture-of-experts layer with M rows in all."""
    b = BF16
    E = experts
    k = {
        # x, W1 in; preact [M,2H] and h [M,H] out
        "fwd_preact": b * (M * D + E * 2 * H * D + 2 * M * H + M * H),
        # h, W2 in; y out
        "fwd_down": b * (M * H + E * Dout * H + M * Dout),
        # dy, W2, preact in; grad_preact [M,2H] and h [M,H] out
        "bwd_grad_h": b * (M * Dout + E * Dout * H + 2 * M * H + 2 * M * H + M * H),
        "bwd_dW2": b * (M * Dout + M * H + E * Dout * H),
        "bwd_dx": b * (2 * M * H + E * 2 * H * D + M * D),
        "bwd_dW1": b * (2 * M * H + M * D + E * 2 * H * D),
    }
    k["bwd_gemms"] = k["bwd_dW2"] + k["bwd_dx"] + k["bwd_dW1"]
    return k
