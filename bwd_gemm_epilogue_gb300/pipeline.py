"""Training steps on host-resident batches, with host<->device copies overlapped.

``HostStepRunner`` runs the block's forward + backward (through the C ABI) on
inputs that live in pinned host memory and returns the results to pinned host
memory, every step.  Three CUDA streams and two device-side buffer sets let the
host->device copy of step i+1 and the device->host copy of step i-1 run while
step i computes:

    h2d stream      copy in (x, W1, W2, dy) of step i+1 into buffer (i+1) % 2
    compute stream  swiglu_mlp_fwd + swiglu_mlp_bwd (or the MoE layer's
                    swiglu_moe_fwd + swiglu_moe_bwd) of step i on buffer i % 2
    d2h stream      copy out (y, dx, dW1, dW2) of step i-1 from buffer (i-1) % 2

Events order the reuse of each buffer: inputs of a buffer are overwritten only
after the compute that read them finished, outputs only after their copy-out
finished.  Device memory: two sets of inputs and outputs plus one preact and
the two workspaces (about 3.7 GB at the target shape).
"""
from __future__ import annotations

import torch

from . import binding


class HostStepRunner:
    """counts: per-expert row counts for a mixture-of-experts layer (swiglu_moe_*;
    W1 [E,2H,D], W2 [E,Dout,H] and their gradients per expert, M = sum(counts));
    None for one block."""

    def __init__(self, M: int, D: int, H: int, Dout: int, device=None, residual: bool = False, counts=None):
        self.dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        self.shape = (M, D, H, Dout)
        self.counts = None if counts is None else [int(c) for c in counts]
        if self.counts is not None and (sum(self.counts) != M or residual):
            raise ValueError("counts must sum to M; the MoE layer has no residual variant")
        E = () if counts is None else (len(self.counts),)
        bf = dict(dtype=torch.bfloat16, device=self.dev)
        self.inp = [dict(x=torch.empty(M, D, **bf), W1=torch.empty(*E, 2 * H, D, **bf),
                         W2=torch.empty(*E, Dout, H, **bf), dy=torch.empty(M, Dout, **bf)) for _ in range(2)]
        self.out = [dict(y=torch.empty(M, Dout, **bf), dx=torch.empty(M, D, **bf),
                         dW1=torch.empty(*E, 2 * H, D, **bf), dW2=torch.empty(*E, Dout, H, **bf)) for _ in range(2)]
        self.preact = torch.empty(M, 2 * H, **bf)
        self.residual = residual      # residual block: y = x + MLP(x), dx += dy
        if self.counts is None:
            fb = binding.swiglu_mlp_fwd_workspace_size(M, D, H, Dout)
            bb = binding.swiglu_mlp_bwd_workspace_size(M, D, H, Dout)
        else:
            fb = binding.swiglu_moe_fwd_workspace_size(self.counts, D, H, Dout)
            bb = binding.swiglu_moe_bwd_workspace_size(self.counts, D, H, Dout)
        self.ws_f = torch.empty(max(16, fb), dtype=torch.uint8, device=self.dev)
        self.ws_b = torch.empty(max(16, bb), dtype=torch.uint8, device=self.dev)
        self.s_h2d = torch.cuda.Stream(self.dev)
        self.s_cmp = torch.cuda.Stream(self.dev)
        self.s_d2h = torch.cuda.Stream(self.dev)
        ev = lambda: torch.cuda.Event()  # noqa: E731
        self.h2d_done = [ev(), ev()]
        self.cmp_done = [ev(), ev()]
        self.d2h_done = [ev(), ev()]
        self._used = [False, False]

    @staticmethod
    def bytes_in(host_in) -> int:
        return sum(t.numel() * t.element_size() for t in host_in.values())

    @staticmethod
    def bytes_out(host_out) -> int:
        return sum(t.numel() * t.element_size() for t in host_out.values())

    def _copy_in(self, i, host_in):
        b = i % 2
        with torch.cuda.stream(self.s_h2d):
            if self._used[b]:
                self.s_h2d.wait_event(self.cmp_done[b])
            for k, t in self.inp[b].items():
                t.copy_(host_in[k], non_blocking=True)
            self.h2d_done[b].record(self.s_h2d)

    def _compute(self, i):
        b = i % 2
        d, o = self.inp[b], self.out[b]
        with torch.cuda.stream(self.s_cmp):
            self.s_cmp.wait_event(self.h2d_done[b])
            if self._used[b]:
                self.s_cmp.wait_event(self.d2h_done[b])
            if self.counts is None:
                binding.swiglu_mlp_fwd(d["x"], d["W1"], d["W2"], self.preact, o["y"], self.ws_f,
                                       residual=self.residual)
                binding.swiglu_mlp_bwd(d["x"], d["W1"], d["W2"], self.preact, d["dy"], o["dx"], o["dW1"],
                                       o["dW2"], self.ws_b, residual=self.residual)
            else:
                binding.swiglu_moe_fwd(d["x"], d["W1"], d["W2"], self.counts, self.preact, o["y"], self.ws_f)
                binding.swiglu_moe_bwd(d["x"], d["W1"], d["W2"], self.preact, d["dy"], self.counts, o["dx"],
                                       o["dW1"], o["dW2"], self.ws_b)
            self.cmp_done[b].record(self.s_cmp)
        self._used[b] = True

    def _copy_out(self, i, host_out):
        b = i % 2
        with torch.cuda.stream(self.s_d2h):
            self.s_d2h.wait_event(self.cmp_done[b])
            for k, t in self.out[b].items():
                host_out[k].copy_(t, non_blocking=True)
            self.d2h_done[b].record(self.s_d2h)

    def run(self, host_ins, host_outs):
        """Run len(host_ins) steps.  host_ins[i]: dict x, W1, W2, dy (pinned CPU bf16);
        host_outs[i]: dict y, dx, dW1, dW2 (pinned CPU bf16), filled on return.
        Returns after every copy-out has been enqueued; synchronise the device (or
        the d2h stream) before reading host_outs."""
        n = len(host_ins)
        if n == 0:
            return
        self._copy_in(0, host_ins[0])
        for i in range(n):
            if i + 1 < n:
                self._copy_in(i + 1, host_ins[i + 1])
            self._compute(i)
            self._copy_out(i, host_outs[i])

    def synchronize(self):
        self.s_d2h.synchronize()
        self.s_cmp.synchronize()
        self.s_h2d.synchronize()
