/*
 * swiglu_moe.h -- C ABI of the mixture-of-experts SwiGLU layer (same library as
 * swiglu_mlp.h, same status codes and conventions).
 *
 * "Lesson 24: MLP, GEMM and operator fusion in the Transformer"
 * (lincklin.cn/blog/gpu-architecture/24_transformer_mlp_gemm_fusion/):
 * section 41 -- each expert of an MoE layer is an MLP of its own and a router
 * sends every token to an expert; sections 42-43 -- the experts' GEMMs differ
 * only in their row counts, so they run as one grouped launch whose blocks are
 * scheduled over the tiles of all experts.
 *
 * Here every expert e is the SwiGLU block of swiglu_mlp.h with its own weights
 * W1[e] [2H, D], W2[e] [Dout, H] and its own rows.  The tokens come already
 * grouped by expert (routing, sorting and packing happen before this layer):
 *
 *   counts[E]      host array, counts[e] >= 0 rows for expert e;
 *                  off[e] = counts[0] + ... + counts[e-1], T = off[E] < 2^31
 *   x  [T, D]      rows off[e] .. off[e] + counts[e] - 1 belong to expert e
 *   W1 [E, 2H, D], W2 [E, Dout, H]   stacked expert weights
 *   preact [T, 2H], y [T, Dout], dx [T, D]            per-row outputs
 *   dW1 [E, 2H, D], dW2 [E, Dout, H]                  per-expert outputs
 *
 * Each of the block's steps (x @ W1^T + SwiGLU; h @ W2^T; dy @ W2 fused with the
 * SwiGLU backward; dW2, dx and dW1) runs as ONE persistent launch over all
 * experts: a table of per-expert problems (tensor maps clipped to the expert's
 * rows, sizes) is copied to the workspace in stream order, and the CTA pairs walk
 * a host tile list that balances the experts' tiles longest-first.  Rows are not
 * padded: an expert's last tile reads zeros past its rows and stores only its own.
 * An expert with no rows contributes no tiles; its dW1[e] and dW2[e] are zeroed.
 *
 * Unlike the entry points of swiglu_mlp.h, these keep a small ring of pinned host
 * buffers per device for the problem tables (allocated on first use, kept for
 * the process's life); a call waits on the host only when the ring wraps onto a
 * table whose copy has not completed yet (eight calls back).
 * E must be in 1..682; D, H, Dout positive multiples of 8; pointers 16-byte
 * aligned; counts must not be NULL.
 */
#ifndef SWIGLU_MOE_H
#define SWIGLU_MOE_H

#include "swiglu_mlp.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Workspace bytes of swiglu_moe_fwd: h [T, H] bf16 and two problem tables.
 * 0 when the arguments are invalid. */
size_t swiglu_moe_fwd_workspace_size(const int64_t* counts, int64_t E, int64_t D, int64_t H, int64_t Dout);

/* Workspace bytes of swiglu_moe_bwd: h [T, H], grad_preact [T, 2H] (bf16, the same
 * layout as swiglu_mlp_bwd's workspace: h first, grad_preact at the next 256-byte
 * boundary) and two problem tables.  0 when the arguments are invalid. */
size_t swiglu_moe_bwd_workspace_size(const int64_t* counts, int64_t E, int64_t D, int64_t H, int64_t Dout);

/* Forward of every expert on its rows: preact and y (h is transient, in the workspace). */
swiglu_status swiglu_moe_fwd(const void* x, const void* W1, const void* W2, void* preact, void* y,
                             const int64_t* counts, int64_t E, int64_t D, int64_t H, int64_t Dout,
                             void* workspace, size_t workspace_bytes, void* stream);

/* Backward of every expert on its rows: dx, dW1, dW2 from the saved preact and dy.
 * T = 0 only zeroes dW1 and dW2 (x, preact, dy, dx and workspace may then be NULL). */
swiglu_status swiglu_moe_bwd(const void* x, const void* W1, const void* W2, const void* preact,
                             const void* dy, void* dx, void* dW1, void* dW2,
                             const int64_t* counts, int64_t E, int64_t D, int64_t H, int64_t Dout,
                             void* workspace, size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SWIGLU_MOE_H */
