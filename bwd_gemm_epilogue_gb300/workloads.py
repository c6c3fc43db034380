"""Seeded synthetic inputs for the SwiGLU MLP block.

This module is shared by the CUDA path's tests/benchmark and by the oracle's
tests; it holds no arithmetic of the method -- only random draws, scaling by
the fan-in rule and bf16 rounding of the draws.  Everything is generated on
the CPU with ``torch.Generator`` so both sides see identical bf16 bits.

Workloads (shapes from the pages' target configuration and the usual LLaMA-7B
prefill/decode shapes; distributions: activations and dy ~ N(0, 1), weights
~ N(0, 1/fan_in)):

  tiny     M=128,   D=256,  H=512,   Dout=256   seed 0 (gate column 0 swept
                                                over [-20, 20], see below)
  decode   M=16,    D=4096, H=11008, Dout=4096  seed 1
  prefill  M=4096,  D=4096, H=11008, Dout=4096  seed 2
  target   M=11136, D=3584, H=14336, Dout=3584  seed 3
  stack4   4 layers of the target block; x, dy from seed 4, layer l's weights
           from seed 100 + l

The gate sweep of the tiny workload sets x[:, 0] = linspace(-20, 20, M) and
makes W1's first gate row the unit vector e_0, so that preact[:, H] = x[:, 0]
exactly and the sigmoid saturates at both ends.

Mixture-of-experts workloads (tokens already grouped by expert; expert e owns
rows [off_e, off_e + counts[e]); W1 [E, 2H, D], W2 [E, Dout, H]):

  moe_tiny  E=4,  counts 32/120/8/64 (the per-expert token counts printed in
            "Lesson 24: MLP, GEMM and operator fusion in the Transformer",
            section 42), D=256, H=512, Dout=256                      seed 5
  moe8      E=8,  T=16384 routed rows (8192 tokens, two experts each),
            D=Dout=4096, H=14336 (Mixtral-8x7B expert shape)          seed 6
  moe64     E=64, T=24576 routed rows (4096 tokens, six experts each),
            D=Dout=2048, H=1408 (fine-grained experts), two experts
            receive no tokens                                         seed 7

Routed counts: expert probabilities uniform on the simplex (normalised
exponential draws; the experts listed as empty get probability 0), T draws
from them, counted per expert.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Shape:
    M: int
    D: int
    H: int
    Dout: int


CONFIGS = {
    "tiny": dict(shape=Shape(128, 256, 512, 256), seed=0, layers=1, gate_sweep=True),
    "decode": dict(shape=Shape(16, 4096, 11008, 4096), seed=1, layers=1, gate_sweep=False),
    "prefill": dict(shape=Shape(4096, 4096, 11008, 4096), seed=2, layers=1, gate_sweep=False),
    "target": dict(shape=Shape(11136, 3584, 14336, 3584), seed=3, layers=1, gate_sweep=False),
    "stack4": dict(shape=Shape(11136, 3584, 14336, 3584), seed=4, layers=4, gate_sweep=False),
}

# Stream ids: each tensor comes from its own generator so any one of them can be
# drawn without drawing the others.
_X, _W1, _W2, _DY, _PREACT = 0, 1, 2, 3, 4


def _gen(seed: int, stream: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed * 1000 + stream)
    return g


def normal_bf16(shape, std: float, seed: int, stream: int) -> torch.Tensor:
    """N(0, std^2) drawn in fp32 on the CPU, then rounded to bf16 (round-to-nearest-even)."""
    t = torch.randn(tuple(shape), generator=_gen(seed, stream), dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(torch.bfloat16)


def make_weights(s: Shape, seed: int, gate_sweep: bool = False):
    """W1 [2H, D] ~ N(0, 1/D) (rows [left | gate]) and W2 [Dout, H] ~ N(0, 1/H)."""
    W1 = normal_bf16((2 * s.H, s.D), s.D ** -0.5, seed, _W1)
    W2 = normal_bf16((s.Dout, s.H), s.H ** -0.5, seed, _W2)
    if gate_sweep:
        W1[s.H].zero_()
        W1[s.H, 0] = 1.0
    return W1, W2


def make_activations(s: Shape, seed: int, gate_sweep: bool = False):
    """x [M, D] ~ N(0, 1) and dy [M, Dout] ~ N(0, 1)."""
    x = normal_bf16((s.M, s.D), 1.0, seed, _X)
    dy = normal_bf16((s.M, s.Dout), 1.0, seed, _DY)
    if gate_sweep and s.M > 0:
        x[:, 0] = torch.linspace(-20.0, 20.0, s.M, dtype=torch.float32).to(torch.bfloat16)
    return x, dy


def make_preact(s: Shape, seed: int, gate_sweep: bool = False) -> torch.Tensor:
    """A stand-in for the saved preact [M, 2H] ~ N(0, 1) (the forward's output
    distribution under the fan-in weight scaling), for backward-only tests at
    sizes where the oracle cannot run the forward."""
    p = normal_bf16((s.M, 2 * s.H), 1.0, seed, _PREACT)
    if gate_sweep and s.M > 0:
        p[:, s.H] = torch.linspace(-20.0, 20.0, s.M, dtype=torch.float32).to(torch.bfloat16)
    return p


def make_block(name_or_shape, seed: int | None = None, gate_sweep: bool | None = None):
    """x, W1, W2, dy for one block: a named workload or an explicit Shape."""
    if isinstance(name_or_shape, str):
        cfg = CONFIGS[name_or_shape]
        s = cfg["shape"]
        seed = cfg["seed"] if seed is None else seed
        gate_sweep = cfg["gate_sweep"] if gate_sweep is None else gate_sweep
    else:
        s = name_or_shape
        seed = 0 if seed is None else seed
        gate_sweep = bool(gate_sweep)
    x, dy = make_activations(s, seed, gate_sweep)
    W1, W2 = make_weights(s, seed, gate_sweep)
    return s, x, W1, W2, dy


def make_stack(name: str = "stack4"):
    """x, dy and per-layer (W1, W2) for the layered workload."""
    cfg = CONFIGS[name]
    s = cfg["shape"]
    x, dy = make_activations(s, cfg["seed"])
    layers = [make_weights(s, 100 + l) for l in range(cfg["layers"])]
    return s, x, dy, layers


MOE_CONFIGS = {
    "moe_tiny": dict(E=4, counts=(32, 120, 8, 64), D=256, H=512, Dout=256, seed=5, empty=0),
    "moe8": dict(E=8, T=16384, D=4096, H=14336, Dout=4096, seed=6, empty=0),
    "moe64": dict(E=64, T=24576, D=2048, H=1408, Dout=2048, seed=7, empty=2),
}
_COUNTS = 5


def moe_counts(T: int, E: int, seed: int, empty: int = 0) -> list:
    """Per-expert row counts summing to T (see the module docstring); the last
    `empty` experts receive none."""
    g = _gen(seed, _COUNTS)
    w = -torch.log(torch.rand(E, generator=g, dtype=torch.float64))
    w[E - empty:] = 0.0
    picks = torch.multinomial(w / w.sum(), T, replacement=True, generator=g)
    return [int(v) for v in torch.bincount(picks, minlength=E)]


def make_moe(name: str):
    """counts, x [T, D], W1 [E, 2H, D], W2 [E, Dout, H], dy [T, Dout] for a named MoE workload."""
    cfg = MOE_CONFIGS[name]
    E, D, H, Dout, seed = cfg["E"], cfg["D"], cfg["H"], cfg["Dout"], cfg["seed"]
    counts = list(cfg["counts"]) if "counts" in cfg else moe_counts(cfg["T"], E, seed, cfg["empty"])
    s = Shape(sum(counts), D, H, Dout)
    x, dy = make_activations(s, seed)
    W1 = normal_bf16((E, 2 * H, D), D ** -0.5, seed, _W1)
    W2 = normal_bf16((E, Dout, H), H ** -0.5, seed, _W2)
    return counts, x, W1, W2, dy


def pow2_scale(t: torch.Tensor, fmax: float = 448.0) -> float:
    """The smallest power of two s with max|t| / s <= fmax (per-tensor FP8 scale)."""
    import math
    amax = float(t.abs().max()) if t.numel() else 0.0
    return 2.0 ** math.ceil(math.log2(amax / fmax)) if amax > 0 else 1.0


def to_e4m3(t: torch.Tensor, s: float) -> torch.Tensor:
    """t / s as FP8 E4M3 (torch's conversion: round to nearest even)."""
    return (t.float() / s).to(torch.float8_e4m3fn)


def make_fp8_block(s: Shape, seed: int, s_h: float = 1.0 / 32):
    """FP8 inputs of the block: x8, W1_8, W2_8 (E4M3) and per-tensor power-of-two
    scales {s_x, s_w1, s_w2, s_h}, from the same draws as make_block (x ~ N(0,1),
    weights ~ N(0, 1/fan_in)).  s_h, the scale h is quantised with, is fixed: with
    preact ~ N(0,1) a few of the largest h saturate at 448 * s_h = 14."""
    x = torch.randn((s.M, s.D), generator=_gen(seed, _X), dtype=torch.float32)
    W1 = torch.randn((2 * s.H, s.D), generator=_gen(seed, _W1), dtype=torch.float32) * s.D ** -0.5
    W2 = torch.randn((s.Dout, s.H), generator=_gen(seed, _W2), dtype=torch.float32) * s.H ** -0.5
    sc = {"s_x": pow2_scale(x), "s_w1": pow2_scale(W1), "s_w2": pow2_scale(W2), "s_h": float(s_h)}
    return to_e4m3(x, sc["s_x"]), to_e4m3(W1, sc["s_w1"]), to_e4m3(W2, sc["s_w2"]), sc
