"""GB300-native SwiGLU MLP block: forward, and a backward whose activation-gradient
GEMM grad_h = dy @ W2 carries the SwiGLU backward in its epilogue; also the residual
block, a mixture-of-experts layer of such blocks and an FP8 forward.

The compute path is a C-ABI shared library of hand-written sm_103a kernels
(``csrc/``, declared in ``include/swiglu_mlp.h`` and ``include/swiglu_moe.h``);
``binding`` marshals arguments to it with ctypes.  Importing this package does not
load the library; the first call into ``binding`` does, and raises if it has not
been built.  ``stack`` (stacked blocks) and ``pipeline`` (steps on host batches)
sit on top of ``binding``.
"""
__all__ = ["binding", "workloads", "ledger", "stack", "pipeline"]
