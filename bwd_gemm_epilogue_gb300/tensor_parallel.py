"""Tensor-parallel SwiGLU block: column-parallel first projection, row-parallel down
projection ("Lesson 24: MLP, GEMM and operator fusion in the Transformer", lincklin.cn,
section 33), with the reduction of each row chunk overlapped with the down projection of
the next (section 39).

Rank r of `world` owns the hidden units J = [r * Hs, (r + 1) * Hs) with Hs = H / world:
W1 rows J and H + J (the left and gate rows of the same hidden units, so its SwiGLU is
local) and W2 columns J.  Its forward gives a partial y, its backward a partial dx; the
ranks add them up with one collective each.  The weight gradients of a shard are
complete on its rank (no reduction), and so is its saved preact [M, 2 * Hs].

On CUDA tensors the shard products run in the library (swiglu_mlp_tp_fwd / _bwd, which
record an event per finished row chunk of y and one when dx is final) and the
collectives run on a communication stream that waits for those events, so chunk c is
reduced while chunk c + 1 is computed and dx is reduced while dW1 and dW2 are computed.
`compute` replaces the library for CPU tensors (the multi-rank tests run the gloo
backend on the host with a CPU implementation of the shard products).
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from . import binding


def shard_bounds(H: int, world: int, rank: int) -> tuple[int, int]:
    """(j0, Hs): the first hidden unit and the number of hidden units of `rank`."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} of world {world}")
    if H % world or (H // world) % 8:
        raise ValueError(f"H = {H} must split into {world} shards of a multiple of 8 hidden units")
    Hs = H // world
    return rank * Hs, Hs


class LibraryShardCompute:
    """The shard products on the GPU, through the C ABI."""

    def chunk_rows(self, M: int, n_chunks: int) -> int:
        return binding.swiglu_mlp_tp_chunk_rows(M, n_chunks)

    def fwd(self, x, W1_shard, W2_shard, n_chunks, chunk_events):
        return binding.swiglu_mlp_tp_fwd(x, W1_shard, W2_shard, n_chunks=n_chunks, chunk_events=chunk_events)

    def bwd(self, x, W1_shard, W2_shard, preact, dy, dx_event):
        return binding.swiglu_mlp_tp_bwd(x, W1_shard, W2_shard, preact, dy, dx_event=dx_event)


class TensorParallelSwiGLU:
    """One rank's part of a tensor-parallel SwiGLU block.

    W1_shard [2*Hs, D] (rows J then H + J) and W2_shard [Dout, Hs] (columns J), e.g. from
    binding.swiglu_mlp_tp_shard_pack.  `group`: the process group of the ranks that share
    the block (None: the default group, or a single rank without torch.distributed).
    reduce = "all_reduce": every rank gets the whole y and dx; "reduce_scatter": the sum
    of row chunk c lands on rank c % world (the others keep their partial sums there).
    """

    def __init__(self, W1_shard, W2_shard, group=None, n_chunks: int = 4, reduce: str = "all_reduce",
                 compute=None):
        if reduce not in ("all_reduce", "reduce_scatter"):
            raise ValueError(f"reduce: {reduce!r}")
        self.W1, self.W2 = W1_shard, W2_shard
        self.group = group
        self.n_chunks = max(1, int(n_chunks))
        self.reduce = reduce
        self.compute = compute if compute is not None else LibraryShardCompute()
        self.distributed = dist.is_available() and dist.is_initialized()
        self.world = dist.get_world_size(group) if self.distributed else 1
        self.rank = dist.get_rank(group) if self.distributed else 0
        self.comm = torch.cuda.Stream(W1_shard.device) if W1_shard.is_cuda else None

    # ------------------------------------------------------------------ collectives
    def owner(self, c: int) -> int:
        """Rank (in the group) that receives the sum of row chunk c under reduce_scatter."""
        return c % self.world

    def _reduce_rows(self, t, c: int, r0: int, r1: int):
        """Start the reduction of rows [r0, r1) (chunk c) of t; returns a work handle or None."""
        if not self.distributed or self.world == 1 or r1 <= r0:
            return None
        part = t[r0:r1]
        if self.reduce == "all_reduce":
            return dist.all_reduce(part, group=self.group, async_op=True)
        dst = self.owner(c)
        if self.group is not None:
            dst = dist.get_global_rank(self.group, dst)
        return dist.reduce(part, dst=dst, group=self.group, async_op=True)

    def _chunks(self, M: int):
        rows = self.compute.chunk_rows(M, self.n_chunks)
        out = []
        for c in range(self.n_chunks):
            r0 = c * rows
            out.append((r0, min(M, r0 + rows)) if rows > 0 and r0 < M else (M, M))
        return out

    # ------------------------------------------------------------------ forward / backward
    def forward(self, x):
        """Returns (y [M, Dout] summed over the ranks (see `reduce`), preact_shard [M, 2*Hs])."""
        M = x.shape[0]
        chunks = self._chunks(M)
        if x.is_cuda:
            events = [torch.cuda.Event() for _ in chunks]
            preact, y = self.compute.fwd(x, self.W1, self.W2, self.n_chunks, events)
            works = []
            cur = torch.cuda.current_stream(x.device)
            # the communication stream waits for each chunk's event only (not for the whole
            # forward), so the reduction of chunk c overlaps the down projection of chunk c+1
            with torch.cuda.stream(self.comm):
                for c, ((r0, r1), ev) in enumerate(zip(chunks, events)):
                    self.comm.wait_event(ev)   # chunk c of y is final
                    works.append(self._reduce_rows(y, c, r0, r1))
            for w in works:
                if w is not None:
                    w.wait()
            cur.wait_stream(self.comm)
            y.record_stream(self.comm)
        else:
            preact, y = self.compute.fwd(x, self.W1, self.W2, self.n_chunks, None)
            for c, (r0, r1) in enumerate(chunks):
                w = self._reduce_rows(y, c, r0, r1)
                if w is not None:
                    w.wait()
        return y, preact

    def backward(self, x, preact, dy):
        """Returns (dx [M, D] summed over the ranks, dW1_shard [2*Hs, D], dW2_shard [Dout, Hs])."""
        M = x.shape[0]
        if x.is_cuda:
            ev = torch.cuda.Event()
            dx, dW1, dW2 = self.compute.bwd(x, self.W1, self.W2, preact, dy, ev)
            cur = torch.cuda.current_stream(x.device)
            works = []
            with torch.cuda.stream(self.comm):
                self.comm.wait_event(ev)   # dx final; dW1 / dW2 still computing on `cur`
                for c, (r0, r1) in enumerate(self._chunks(M)):
                    works.append(self._reduce_rows(dx, c, r0, r1))
            for w in works:
                if w is not None:
                    w.wait()
            cur.wait_stream(self.comm)
            dx.record_stream(self.comm)
        else:
            dx, dW1, dW2 = self.compute.bwd(x, self.W1, self.W2, preact, dy, None)
            for c, (r0, r1) in enumerate(self._chunks(M)):
                w = self._reduce_rows(dx, c, r0, r1)
                if w is not None:
                    w.wait()
        return dx, dW1, dW2
