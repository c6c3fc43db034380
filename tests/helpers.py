"""Shared test helpers: tolerance check, library build/load."""
import os
import re

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# Per-tensor parity bar: relative Frobenius error <= 5e-3 and max abs error <= 2e-2 * max|oracle|.
REL_FRO = 5e-3
MAX_ABS_FRAC = 2e-2


def parity(gpu, ref, name=""):
    """Assert the parity bar between a GPU tensor (any dtype) and an fp64 oracle array."""
    g = gpu.detach().float().cpu().double().numpy() if isinstance(gpu, torch.Tensor) else np.asarray(gpu, np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, f"{name}: shape {g.shape} vs {r.shape}"
    assert np.all(np.isfinite(g)), f"{name}: non-finite values"
    nr = np.linalg.norm(r)
    err = np.linalg.norm(g - r)
    rel = err / nr if nr > 0 else err
    mx = np.max(np.abs(r)) if r.size else 0.0
    worst = np.max(np.abs(g - r)) if r.size else 0.0
    assert rel <= REL_FRO, f"{name}: relative Frobenius error {rel:.3e} > {REL_FRO}"
    assert worst <= MAX_ABS_FRAC * mx + 1e-30, f"{name}: max abs error {worst:.3e} > {MAX_ABS_FRAC} * {mx:.3e}"
    return rel, worst


def header_functions():
    """Names of the functions the headers under include/ declare."""
    names = set()
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if h.endswith(".h"):
            src = open(os.path.join(ROOT, "include", h)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(swiglu_(?:mlp|moe)_\w+)\s*\(", src))
    return sorted(names)


def ensure_library():
    from bwd_gemm_epilogue_gb300 import build
    return build.build()
