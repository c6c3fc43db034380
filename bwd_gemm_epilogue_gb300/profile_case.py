"""Run one kernel of the block on a medium case, for ncu captures.

    python -m bwd_gemm_epilogue_gb300.profile_case --kernel bwd_grad_h --M 4096 --iters 3

Inputs are the target block's widths (D = Dout = 3584, H = 14336) with a smaller
token count M, so the operands still exceed the 129 MB L2 while the whole case
holds well under a few GB of device memory.  Each iteration launches one kernel
of the chosen kind (the fused segment, the forward GEMM with its SwiGLU epilogue,
or one of the plain GEMMs) through the C ABI, or the whole forward ("fwd": two
launches) or backward ("bwd": the fused kernel, then the grouped dW2/dx/dW1).
"fp8_fwd" runs the FP8 forward at the same widths; "moe_fwd" / "moe_bwd" run a
named mixture-of-experts workload (--workload, full size: a few GB) forward or
backward, each step one grouped launch over the experts.
"""
from __future__ import annotations

import argparse

import torch

from . import binding, workloads
from .workloads import Shape

KERNELS = ("fwd_preact", "fwd_down", "bwd_grad_h", "bwd_dW2", "bwd_dx", "bwd_dW1", "fwd", "bwd", "fp8_fwd",
           "moe_fwd", "moe_bwd")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--kernel", choices=KERNELS, default="bwd_grad_h")
    ap.add_argument("--M", type=int, default=4096)
    ap.add_argument("--D", type=int, default=3584)
    ap.add_argument("--H", type=int, default=14336)
    ap.add_argument("--Dout", type=int, default=3584)
    ap.add_argument("--iters", type=int, default=3)
    ap.add_argument("--workload", default="moe64", choices=sorted(workloads.MOE_CONFIGS))
    a = ap.parse_args()
    dev = torch.device("cuda", 0)
    if a.kernel.startswith("moe_"):
        counts, x, W1, W2, dy = (t if isinstance(t, list) else t.to(dev) for t in workloads.make_moe(a.workload))
        T, H = x.shape[0], W2.shape[2]
        preact = workloads.make_preact(Shape(T, x.shape[1], H, W2.shape[1]), seed=7).to(dev)
        for _ in range(a.iters):
            if a.kernel == "moe_fwd":
                binding.swiglu_moe_fwd(x, W1, W2, counts)
            else:
                binding.swiglu_moe_bwd(x, W1, W2, preact, dy, counts)
        st = binding.swiglu_mlp_device_status(dev)
        if st != 0:
            raise SystemExit(f"device status {binding.swiglu_mlp_strerror(st)}")
        print("ok", a.kernel, a.workload, len(counts), "experts", T, "rows")
        return
    s = Shape(a.M, a.D, a.H, a.Dout)
    if a.kernel == "fp8_fwd":
        x8, W1_8, W2_8, sc = (t if isinstance(t, dict) else t.to(dev) for t in workloads.make_fp8_block(s, seed=7))
        for _ in range(a.iters):
            binding.swiglu_mlp_fwd_fp8(x8, W1_8, W2_8, store_preact=False, **sc)
        st = binding.swiglu_mlp_device_status(dev)
        if st != 0:
            raise SystemExit(f"device status {binding.swiglu_mlp_strerror(st)}")
        print("ok", a.kernel, s)
        return
    _, x, W1, W2, dy = workloads.make_block(s, seed=7)
    preact = workloads.make_preact(s, seed=7)
    x, W1, W2, dy, preact = (t.to(dev) for t in (x, W1, W2, dy, preact))
    h = torch.empty(s.M, s.H, dtype=torch.bfloat16, device=dev)
    gp = torch.empty(s.M, 2 * s.H, dtype=torch.bfloat16, device=dev)
    for _ in range(a.iters):
        k = a.kernel
        if k == "bwd_grad_h":
            binding.swiglu_mlp_fused_grad_preact(dy, W2, preact, gp, h)
        elif k == "fwd_preact":
            # the forward also launches the down projection; profile with -k to pick one
            binding.swiglu_mlp_fwd(x, W1, W2)
        elif k == "fwd_down":
            binding.swiglu_mlp_gemm_bf16(h, W2, s.M, s.Dout, s.H, False, False)
        elif k == "bwd_dW2":
            binding.swiglu_mlp_gemm_bf16(dy, h, s.Dout, s.H, s.M, True, True)
        elif k == "bwd_dx":
            binding.swiglu_mlp_gemm_bf16(gp, W1, s.M, s.D, 2 * s.H, False, True)
        elif k == "bwd_dW1":
            binding.swiglu_mlp_gemm_bf16(gp, x, 2 * s.H, s.D, s.M, True, True)
        elif k == "fwd":      # x @ W1^T + SwiGLU epilogue, then h @ W2^T
            binding.swiglu_mlp_fwd(x, W1, W2)
        elif k == "bwd":      # fused grad_h + SwiGLU backward, then the grouped dW2 / dx / dW1 launch
            binding.swiglu_mlp_bwd(x, W1, W2, preact, dy)
    st = binding.swiglu_mlp_device_status(dev)
    if st != 0:
        raise SystemExit(f"device status {binding.swiglu_mlp_strerror(st)}")
    print("ok", a.kernel, s)


if __name__ == "__main__":
    main()
