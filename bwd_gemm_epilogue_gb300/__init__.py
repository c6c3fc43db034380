"""GB300-native SwiGLU MLP block: forward, and a backward whose activation-gradient
GEMM grad_h = dy @ W2 carries the SwiGLU backward in its epilogue.

The compute path is a C-ABI shared library of hand-written sm_103a kernels
(``csrc/``, declared in ``include/swiglu_mlp.h``); ``binding`` marshals
arguments to it with ctypes.  Importing this package does not load the library;
the first call into ``binding`` does, and raises if it has not been built.
"""
__all__ = ["binding", "workloads", "ledger"]
