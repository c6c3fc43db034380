/*
 * swiglu_mlp.h -- C ABI of the GB300 (sm_103a) SwiGLU MLP block.
 *
 * The block (notation of the "SwiGLU MLP Drop-H technical report",
 * lgystoic.github.io/notes/swiglu-mlp-drop-h/, "original math" section):
 *
 *   forward   preact = x @ W1^T        x [M,D], W1 [2H,D] with rows [left | gate]
 *             h      = left * silu(gate)    (left = preact[:, :H], gate = preact[:, H:])
 *             y      = h @ W2^T        W2 [Dout,H]
 *   backward  grad_h      = dy @ W2
 *             grad_preact = [grad_h * silu(gate) | grad_h * left * silu'(gate)]
 *             dx  = grad_preact @ W1,  dW1 = grad_preact^T @ x,  dW2 = dy^T @ h
 *
 * The forward keeps preact (saved for the backward) and drops h after the down
 * projection (the report's "drop-h" saved-tensor policy).  The backward computes
 * grad_h = dy @ W2 on the tensor cores and applies the SwiGLU backward in that
 * GEMM's epilogue, recomputing sigma/silu and h from the saved preact, so grad_h
 * never reaches HBM (the fused dout-GEMM + SwiGLU-backward segment of the
 * "SwiGLU MLP forward/backward optimization" note, section 4).
 *
 * Conventions shared by every entry point:
 *  - Every tensor is a dense, row-major bf16 array in device memory, given as a
 *    plain pointer; shapes are given in elements.  The caller owns all memory
 *    (outputs and workspaces included).  The library allocates nothing, frees
 *    nothing and never synchronises, except swiglu_mlp_device_status.
 *  - All work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) of the current CUDA device; a call returns once it is enqueued.
 *  - Inputs are never written (the backward is non-inplace: preact and dy keep
 *    their contents).  Outputs must not alias inputs or each other.
 *  - Pointers must be 16-byte aligned; D, H and Dout must be positive multiples of
 *    8 (TMA row strides are multiples of 16 bytes); M may be any value >= 0, and
 *    M, 2H, D, Dout must stay below 2^31.
 *  - Errors are returned as a swiglu_status; argument errors are detected before
 *    anything is enqueued.  A kernel that stops making progress (a bounded device
 *    wait ran out) records it in a device error word, which
 *    swiglu_mlp_device_status reads.
 */
#ifndef SWIGLU_MLP_H
#define SWIGLU_MLP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SWIGLU_OK = 0,
    SWIGLU_ERR_INVALID_ARG = 1,        /* null pointer, negative size, aliasing */
    SWIGLU_ERR_UNSUPPORTED_SHAPE = 2,  /* D, H, Dout not positive multiples of 8, or too large */
    SWIGLU_ERR_MISALIGNED = 3,         /* a pointer is not 16-byte aligned */
    SWIGLU_ERR_WORKSPACE_TOO_SMALL = 4,
    SWIGLU_ERR_LAUNCH = 5,             /* a kernel launch or tensor-map encode failed */
    SWIGLU_ERR_TIMEOUT = 6,            /* a device-side wait ran out (see swiglu_mlp_device_status) */
    SWIGLU_ERR_CUDA = 7                /* any other CUDA runtime error */
} swiglu_status;

/* Bytes of workspace swiglu_mlp_fwd needs: the transient h [M,H] bf16; for M <= 64
 * also the small-M path's fp32 partial sums of preact^T [2H, M16] and y^T [Dout, M16]
 * (M16 = M rounded up to 16), one plane per K split (the split counts are planned for
 * 152 SMs), each buffer on a 256-byte boundary.  Where the down projection can split
 * tiles (M >= 256, Dout a multiple of 512, H >= 6337, at least 144 tiles of 256 x 512;
 * see swiglu_mlp_split_plan), h is followed by room for their counters and fp32 sums:
 * 20,480 + 80 x 524,288 bytes. */
size_t swiglu_mlp_fwd_workspace_size(int64_t M, int64_t D, int64_t H, int64_t Dout);

/* Bytes of workspace swiglu_mlp_bwd needs: h [M,H] and grad_preact [M,2H], bf16,
 * each starting on a 256-byte boundary; for M <= 64 also the small-M path's fp32
 * partial sums of grad_h^T [H, M16] and dx^T [D, M16], one plane per K split. */
size_t swiglu_mlp_bwd_workspace_size(int64_t M, int64_t D, int64_t H, int64_t Dout);

/*
 * Forward.  Drop-H report, "Forward: save preact, not h".
 *   x [M,D], W1 [2H,D], W2 [Dout,H]           inputs
 *   preact [M,2H]                              output, saved for the backward
 *   y [M,Dout]                                 output
 *   workspace >= swiglu_mlp_fwd_workspace_size bytes; holds h between the two GEMMs.
 * Kernels: x @ W1^T with a SwiGLU epilogue that writes preact and
 * h = bf16(left * bf16(silu(gate))), then y = h @ W2^T.  For M <= 64 tokens
 * (decode) the two products run transposed with the weights as the 128-row MMA
 * operand, split over K into fp32 workspace sums, and small element-wise kernels
 * apply the SwiGLU and round to bf16.  Each K split writes its own fp32 partial and
 * the element-wise kernels add them in a fixed order, so every path returns the same
 * bits on every run.
 */
swiglu_status swiglu_mlp_fwd(const void* x, const void* W1, const void* W2,
                             void* preact, void* y,
                             int64_t M, int64_t D, int64_t H, int64_t Dout,
                             void* workspace, size_t workspace_bytes, void* stream);

/*
 * Backward.  Drop-H report, "Backward: fused h recompute and grad_preact"
 * (backward formulas), with grad_h fused as in the optimization note, section 4.
 *   x [M,D], W1 [2H,D], W2 [Dout,H], preact [M,2H] (from the forward), dy [M,Dout]   inputs
 *   dx [M,D], dW1 [2H,D], dW2 [Dout,H]                                               outputs
 *   workspace >= swiglu_mlp_bwd_workspace_size bytes; on return (once the stream has
 *   run) it holds h [M,H] at offset 0 and grad_preact [M,2H] at the next 256-byte
 *   boundary after h.
 * Kernels: grad_h = dy @ W2 fused with the SwiGLU backward (writes grad_preact and
 * h), then dW2 = dy^T @ h, dx = grad_preact @ W1, dW1 = grad_preact^T @ x (one merged
 * [2H,M] @ [M,D] product) -- these three independent GEMMs share one persistent
 * launch whose tiles are balanced across the SMs.  With M = 0, dW1 and dW2 are set
 * to zero.
 */
swiglu_status swiglu_mlp_bwd(const void* x, const void* W1, const void* W2,
                             const void* preact, const void* dy,
                             void* dx, void* dW1, void* dW2,
                             int64_t M, int64_t D, int64_t H, int64_t Dout,
                             void* workspace, size_t workspace_bytes, void* stream);

/*
 * Residual block y = x + MLP(x) (requires D == Dout): the down projection adds the
 * block input in its epilogue instead of writing MLP(x) and adding it in a separate
 * pass ("Transformer MLP, GEMM and operator fusion" lesson, section 24, residual-add
 * epilogue).  Same arguments, workspace and saved preact as swiglu_mlp_fwd.
 * D != Dout returns SWIGLU_ERR_UNSUPPORTED_SHAPE.
 */
swiglu_status swiglu_mlp_fwd_residual(const void* x, const void* W1, const void* W2,
                                      void* preact, void* y,
                                      int64_t M, int64_t D, int64_t H, int64_t Dout,
                                      void* workspace, size_t workspace_bytes, void* stream);

/*
 * Backward of the residual block: as swiglu_mlp_bwd, with the identity path's dy
 * added to dx in the dx GEMM's epilogue (dx = grad_preact @ W1 + dy); dW1 and dW2
 * are unchanged.  Requires D == Dout.
 */
swiglu_status swiglu_mlp_bwd_residual(const void* x, const void* W1, const void* W2,
                                      const void* preact, const void* dy,
                                      void* dx, void* dW1, void* dW2,
                                      int64_t M, int64_t D, int64_t H, int64_t Dout,
                                      void* workspace, size_t workspace_bytes, void* stream);

/*
 * FP8 forward with a quantising epilogue ("Lesson 24: MLP, GEMM and operator
 * fusion in the Transformer", lincklin.cn, section 26: the 8-bit GEMM's epilogue
 * scales the accumulator, applies the activation, rounds and saturates to the
 * 8-bit output; section 31: 8-bit weights halve the weight traffic).
 *   x8 [M,D], W1_8 [2H,D], W2_8 [Dout,H]  FP8 E4M3 codes (one byte each), with
 *                                         per-tensor scales: x = s_x * x8, ...
 *   preact [M,2H]  optional bf16 output (NULL: not stored) =
 *                  bf16(s_x * s_w1 * (x8 @ W1_8^T))
 *   h8 [M,H]       E4M3 output: sat8(round(h / s_h)), h = left * bf16(silu(gate))
 *                  from the bf16-rounded preact; round to nearest even, finite
 *                  values beyond +-448 saturate to +-448
 *   y [M,Dout]     bf16 output: s_h * s_w2 * (h8 @ W2_8^T)
 * Both products run on the FP8 tensor cores with fp32 accumulators.  Needs D and H
 * multiples of 16 (16-byte rows of FP8), Dout a multiple of 8, positive finite
 * scales (SWIGLU_ERR_INVALID_ARG otherwise).  For M <= 64 tokens (decode) the
 * products stream the FP8 weights transposed and split over K, as in the bf16
 * forward, into fp32 sums held in the workspace; element-wise kernels scale them,
 * apply the SwiGLU, quantise h and cast y.  Larger M needs no workspace.
 */
size_t swiglu_mlp_fwd_fp8_workspace_size(int64_t M, int64_t D, int64_t H, int64_t Dout);

swiglu_status swiglu_mlp_fwd_fp8(const void* x8, const void* W1_8, const void* W2_8,
                                 float s_x, float s_w1, float s_w2, float s_h,
                                 void* preact, void* h8, void* y,
                                 int64_t M, int64_t D, int64_t H, int64_t Dout,
                                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * The fused segment alone: grad_h = dy @ W2 (never stored) and the SwiGLU
 * backward epilogue.  Optimization note, section 4; Drop-H report, fused kernel
 * pseudo-code.
 *   dy [M,Dout], W2 [Dout,H], preact [M,2H]   inputs
 *   grad_preact [M,2H] = [dleft | dgate], h [M,H]   outputs
 */
swiglu_status swiglu_mlp_fused_grad_preact(const void* dy, const void* W2, const void* preact,
                                           void* grad_preact, void* h,
                                           int64_t M, int64_t H, int64_t Dout, void* stream);

/*
 * The plain tcgen05 GEMM the block's other products use:
 *   C [M,N] = A * B^T, bf16 in, fp32 accumulate, bf16 out.
 *   A is [M,K] row-major when a_mn_major = 0, or [K,M] row-major (A^T stored) when 1.
 *   B is [N,K] row-major when b_mn_major = 0, or [K,N] row-major when 1.
 * M, N, K >= 1; the contiguous dimension of each operand and N must be multiples of 8.
 */
swiglu_status swiglu_mlp_gemm_bf16(const void* A, const void* B, void* C,
                                   int64_t M, int64_t N, int64_t K,
                                   int a_mn_major, int b_mn_major, void* stream);

/*
 * Tensor-parallel shards of the block ("Lesson 24: MLP, GEMM and operator fusion in the
 * Transformer", lincklin.cn, section 33, the column-parallel MLP: the first projection
 * split by output columns, the down projection by rows, and y = Y0 + Y1 + ... summed
 * over the ranks; section 39: the reduction overlaps the GEMM).  Rank r owns the hidden
 * units J = [j0, j0 + Hs): W1 rows J (left) and H + J (the matching gate rows), so its
 * SwiGLU needs nothing from the other ranks, and W2 columns J.  A shard is stored packed:
 *   W1_shard [2*Hs, D] = rows J of W1, then rows H + J;   W2_shard [Dout, Hs] = W2[:, J].
 * Its forward and backward are the block's on the shard (H replaced by Hs): preact_shard
 * [M, 2*Hs] = [left_J | gate_J]; y and dx are PARTIAL sums that the caller adds across the
 * ranks (all-reduce or reduce-scatter); the weight gradients are the shard's own, complete.
 * Workspaces: swiglu_mlp_fwd_workspace_size / swiglu_mlp_bwd_workspace_size with H = Hs.
 *
 * swiglu_mlp_tp_shard_pack copies rank r's shard out of the full weights (W1 [2H, D],
 * W2 [Dout, H]); swiglu_mlp_tp_shard_unpack_grads writes a shard's dW1_shard / dW2_shard
 * into the rows J, H + J of a full dW1 and the columns J of a full dW2 (the other entries
 * are left as they are).  Both are stream-ordered device copies.  Need D, H, Dout, Hs
 * multiples of 8, j0 a multiple of 8 and j0 + Hs <= H (SWIGLU_ERR_UNSUPPORTED_SHAPE
 * otherwise).
 */
swiglu_status swiglu_mlp_tp_shard_pack(const void* W1, const void* W2, void* W1_shard, void* W2_shard,
                                       int64_t D, int64_t H, int64_t Dout, int64_t j0, int64_t Hs, void* stream);
swiglu_status swiglu_mlp_tp_shard_unpack_grads(const void* dW1_shard, const void* dW2_shard, void* dW1, void* dW2,
                                               int64_t D, int64_t H, int64_t Dout, int64_t j0, int64_t Hs,
                                               void* stream);

/*
 * Shard forward: preact_shard and the partial y_partial [M, Dout] = h_J @ W2[:, J]^T.
 * The down projection runs in n_chunks row chunks (1..1024) of
 * swiglu_mlp_tp_chunk_rows(M, n_chunks) rows (whole 256-row tiles; the last chunk may be
 * shorter or empty); when chunk_events is not NULL it holds n_chunks cudaEvent_t handles
 * (caller-owned) and event c is recorded once rows of chunk c of y_partial are final, so a
 * communication stream can start reducing chunk c while chunk c+1 is computed.  With more
 * than one chunk, odd chunks run on a second stream the library keeps for the calling
 * thread (forked from `stream` after the first GEMM, joined back into `stream` before the
 * call returns), so that each chunk starts on the SMs the previous one leaves idle; event c
 * is recorded on the stream that computed chunk c, and work enqueued on `stream` after the
 * call sees every chunk.  For M <= 64 (and n_chunks = 1) the forward runs in one piece on
 * `stream` and every event is recorded at its end.
 */
swiglu_status swiglu_mlp_tp_fwd(const void* x, const void* W1_shard, const void* W2_shard, void* preact_shard,
                                void* y_partial, int64_t M, int64_t D, int64_t Hs, int64_t Dout, int n_chunks,
                                void* const* chunk_events, void* workspace, size_t workspace_bytes, void* stream);
int64_t swiglu_mlp_tp_chunk_rows(int64_t M, int n_chunks);

/*
 * Shard backward: dx_partial [M, D] = grad_preact_J @ W1_shard (a partial sum over the
 * ranks), dW1_shard [2*Hs, D] and dW2_shard [Dout, Hs] (complete).  When dx_event (a
 * caller-owned cudaEvent_t) is not NULL, dx is computed by a launch of its own on `stream`
 * and the event is recorded on `stream` when dx_partial is final, while dW1_shard and
 * dW2_shard are computed beside it on a second stream the library keeps for the calling
 * thread (forked from `stream` after the fused kernel, joined back into `stream` before the
 * call returns), so that dx can be reduced across the ranks meanwhile.  With dx_event NULL
 * this is swiglu_mlp_bwd on the shard.
 */
swiglu_status swiglu_mlp_tp_bwd(const void* x, const void* W1_shard, const void* W2_shard, const void* preact_shard,
                                const void* dy, void* dx_partial, void* dW1_shard, void* dW2_shard, int64_t M,
                                int64_t D, int64_t Hs, int64_t Dout, void* dx_event, void* workspace,
                                size_t workspace_bytes, void* stream);

/*
 * Synchronises `stream`, then returns SWIGLU_TIMEOUT if any kernel of this
 * library on the current device gave up a bounded wait since the last call
 * (and clears that record), SWIGLU_ERR_CUDA if the stream reports a CUDA
 * error, else SWIGLU_OK.
 */
swiglu_status swiglu_mlp_device_status(void* stream);

/*
 * Forward without a caller-supplied workspace.  The pages have no counterpart:
 * this is a convenience for callers that cannot allocate device memory (a plugin
 * whose host framework owns all device allocations and offers no scratch hook, a
 * real-time loop that must not call cudaMalloc because it can synchronise the
 * device, a process whose device memory is fixed at start-up).
 *   Same inputs, outputs and results as swiglu_mlp_fwd; h [M,H] is kept in a
 *   fixed array of SWIGLU_MLP_NOALLOC_SCRATCH_BYTES (64 MiB) inside the library's
 *   device memory, which every GPU that loads the library holds until the process
 *   exits.  M*H*2 must not exceed that size (M*H <= 33554432), else
 *   SWIGLU_ERR_WORKSPACE_TOO_SMALL is returned before anything is enqueued.
 *   The call allocates nothing: no cudaMalloc, no cudaFree, no allocating library.
 *   The first call on a device looks up the array's device address (once per
 *   device, with that device current); make that first call before any stream
 *   capture.  All calls share the one array and each overwrites it, so calls whose
 *   work can overlap on the GPU (different streams without ordering) race on it.
 */
#define SWIGLU_MLP_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)
swiglu_status swiglu_mlp_fwd_noalloc(const void* x, const void* W1, const void* W2,
                                     void* preact, void* y,
                                     int64_t M, int64_t D, int64_t H, int64_t Dout, void* stream);

/* Human-readable name of a status. */
const char* swiglu_mlp_strerror(swiglu_status status);

/* Detail of the last failure reported on the calling thread: the CUDA call or
 * check that failed and the CUDA error name.  Empty before the first failure.
 * The string is owned by the library and stays valid until the thread's next
 * failing call. */
const char* swiglu_mlp_last_error_detail(void);

/* Limit of every device-side wait, in nanoseconds (default 4e9).  Process-wide. */
void swiglu_mlp_set_wait_timeout_ns(uint64_t ns);

/* Test hooks, process-wide, default 0.  Bit 0: the GEMMs' TMA producer issues no
 * loads, so the consumers' waits run out and the kernel returns with
 * SWIGLU_ERR_TIMEOUT recorded (used to test the timeout path; no fault).
 * Bit 1: every GEMM uses single-CTA 128-row tiles instead of CTA-pair 256-row
 * tiles.  Bit 2: the backward launches dW2, dx and dW1 separately instead of as
 * one grouped launch.  Bit 3: M <= 64 keeps the 128-row tile path instead of the
 * small-M path.  Bit 4: MoE launches keep CTA-pair tiles even when 128-row tiles
 * would compute fewer padded rows.  Bit 5: plain GEMMs of CTA pairs always use
 * 256 x 256 tiles; bit 6: they use 256 x 512 tiles wherever N > 256 (by default
 * the library picks per launch).  Bit 7: the forward's down projection splits no
 * tiles (see swiglu_mlp_split_plan).  (Every setting computes the same result, except
 * that a split tile adds two fp32 partial sums, so its outputs can differ from the
 * unsplit tile's in the last bit of rounding; the bits exist to test each path.) */
void swiglu_mlp_set_debug_flags(int flags);

/* Test hook (host only; needs no GPU): the tile lists of one K-major GEMM, M x N over K,
 * in 256 x 512 tiles with split tiles, as the forward's down projection runs it on
 * `units` CTA pairs when N is a multiple of 512 and there are at least two rounds of
 * tiles (y = h @ W2^T: N = Dout, K = H).  Whole tiles go round robin for all rounds but
 * the last; the k-blocks of the remaining tiles
 * are divided evenly over the pairs, and a tile that a boundary cuts is shared by two
 * pairs, one summing its first k-blocks, the other the rest, in fp32 (the pair finishing
 * second adds the other's sums and stores the tile).  Writes up to `cap` rows of five
 * int32: pair, tile (raster index), first k-block, end k-block (exclusive), split index
 * (-1 for a whole tile); pairs in order, each pair's entries in the order it runs them.
 * Returns the number of rows (also when above cap; out may be null), or -1 where the
 * forward does not split tiles for this shape. */
int swiglu_mlp_split_plan(int64_t M, int64_t N, int64_t K, int units, int32_t* out, int cap);

/* Tuning knob, process-wide: the width, in 256-column units, of the bands the tile
 * kernels walk their output in (all rows of a band before the next band, so a band's
 * B slabs stay in L2 while the A slabs stream past; 256 x 512 tiles take half as many
 * tiles per band).  0 (the default) = 8.  Any value >= 1 computes the same result. */
void swiglu_mlp_set_raster_band(int n_tiles);

/* Kernel kinds reported by the launch trace. */
typedef enum {
    SWIGLU_KERNEL_FWD_PREACT = 1,   /* x @ W1^T + SwiGLU forward epilogue */
    SWIGLU_KERNEL_FWD_DOWN = 2,     /* y = h @ W2^T */
    SWIGLU_KERNEL_BWD_GRAD_H = 3,   /* dy @ W2 + SwiGLU backward epilogue (the fused segment) */
    SWIGLU_KERNEL_BWD_DW2 = 4,      /* dW2 = dy^T @ h */
    SWIGLU_KERNEL_BWD_DX = 5,       /* dx = grad_preact @ W1 */
    SWIGLU_KERNEL_BWD_DW1 = 6,      /* dW1 = grad_preact^T @ x */
    SWIGLU_KERNEL_GEMM = 7,         /* swiglu_mlp_gemm_bf16 */
    SWIGLU_KERNEL_BWD_GEMMS = 8,    /* dW2, dx and dW1 in one launch (the backward's default) */
    SWIGLU_KERNEL_ELEMENTWISE = 9   /* small-M path: SwiGLU forward/backward or cast of fp32 sums */
} swiglu_kernel_kind;

/*
 * Launch trace for timing individual kernels inside a larger call.  After
 * swiglu_mlp_trace_begin, the i-th kernel this library launches from the calling
 * thread (i < capacity) is bracketed by cudaEventRecord(events[2i]) and
 * cudaEventRecord(events[2i+1]) on its stream, and kinds[i] receives its
 * swiglu_kernel_kind.  `events` holds 2*capacity cudaEvent_t handles created by
 * the caller with timing enabled; `kinds` holds capacity ints; both stay owned by
 * the caller and must outlive the trace.  swiglu_mlp_trace_end stops tracing and
 * returns the number of launches seen (which may exceed capacity; only the first
 * capacity are recorded).  Tracing adds two event records per launch, nothing else.
 */
void swiglu_mlp_trace_begin(void** events, int* kinds, int capacity);
int swiglu_mlp_trace_end(void);

/* ABI version of this header (major * 100 + minor): 200 = the block, its residual
 * variant, the FP8 forward and (swiglu_moe.h) the MoE layer; 201 adds the
 * tensor-parallel shard entry points. */
int swiglu_mlp_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SWIGLU_MLP_H */
