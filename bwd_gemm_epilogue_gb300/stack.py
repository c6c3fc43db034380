"""A stack of SwiGLU MLP blocks: y_l = block_l(y_{l-1}), trained end to end.

Forward keeps, per layer, only what the block's backward needs beyond its
weights: the layer input x_l (which is the previous layer's output, already
kept) and preact_l -- the drop-h saved-tensor policy applied to every layer
("SwiGLU MLP Drop-H technical report", 4-layer stack memory table).  Backward
walks the layers in reverse; each layer's dx is the next (lower) layer's dy.
Every product runs in the library's kernels through the C ABI.
"""
from __future__ import annotations

import torch

from . import binding


class SwiGLUStack:
    def __init__(self, layers, M: int, device=None):
        """layers: list of (W1 [2H,D], W2 [Dout,H]) CUDA bf16 tensors with D == Dout."""
        self.layers = layers
        self.M = M
        W1, W2 = layers[0]
        self.D = W1.shape[1]
        self.H = W2.shape[1]
        self.Dout = W2.shape[0]
        if self.D != self.Dout:
            raise ValueError("a stack needs D == Dout")
        self.dev = W1.device if device is None else torch.device(device)
        bf = dict(dtype=torch.bfloat16, device=self.dev)
        L = len(layers)
        self.acts = [torch.empty(M, self.D, **bf) for _ in range(L + 1)]     # x_0 .. x_L (= y)
        self.preacts = [torch.empty(M, 2 * self.H, **bf) for _ in range(L)]
        self.grads = [(torch.empty(2 * self.H, self.D, **bf), torch.empty(self.Dout, self.H, **bf)) for _ in range(L)]
        self.dacts = [torch.empty(M, self.D, **bf) for _ in range(2)]        # ping-pong dy / dx
        self.ws_f = torch.empty(max(16, binding.swiglu_mlp_fwd_workspace_size(M, self.D, self.H, self.Dout)),
                                dtype=torch.uint8, device=self.dev)
        self.ws_b = torch.empty(max(16, binding.swiglu_mlp_bwd_workspace_size(M, self.D, self.H, self.Dout)),
                                dtype=torch.uint8, device=self.dev)

    def forward(self, x):
        self.acts[0].copy_(x)
        for l, (W1, W2) in enumerate(self.layers):
            binding.swiglu_mlp_fwd(self.acts[l], W1, W2, self.preacts[l], self.acts[l + 1], self.ws_f)
        return self.acts[-1]

    def backward(self, dy):
        """Returns (dx of the stack input, [(dW1_l, dW2_l) for each layer])."""
        cur = dy
        for l in range(len(self.layers) - 1, -1, -1):
            W1, W2 = self.layers[l]
            dW1, dW2 = self.grads[l]
            out = self.dacts[l % 2]
            binding.swiglu_mlp_bwd(self.acts[l], W1, W2, self.preacts[l], cur, out, dW1, dW2, self.ws_b)
            cur = out
        return cur, self.grads

    def saved_activation_bytes(self) -> int:
        """What the forward keeps for the backward beyond the weights: every layer's
        input (x_0 .. x_{L-1}), every preact, and the output."""
        t = self.acts + self.preacts
        return sum(a.numel() * a.element_size() for a in t)

    def backward_peak_bytes(self) -> int:
        """Device memory held at the backward's peak beyond the weights, x and dy (the
        caller's): the saved activations, the backward workspace (h and grad_preact of
        one layer), the dx ping-pong buffers and every layer's weight gradients.  The
        forward's workspace (h) is idle during the backward and not counted."""
        extra = [self.ws_b] + self.dacts + [g for pair in self.grads for g in pair]
        return self.saved_activation_bytes() + sum(a.numel() * a.element_size() for a in extra)
