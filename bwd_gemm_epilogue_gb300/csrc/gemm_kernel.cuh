// gemm_kernel.cuh -- persistent, warp-specialised tcgen05 GEMM for sm_103a with
// the SwiGLU MLP block's epilogues.
//
//   C[M, N] = A[M, K] * B[N, K]^T        bf16 (or FP8 E4M3) in, fp32 accumulate in TMEM
//
// A and B are each either K-major (K contiguous in memory) or MN-major (M or N
// contiguous); the TMA boxes and the UMMA shared-memory descriptors differ, the
// rest of the kernel does not.  Template parameters: EPI (epilogue, below), CG (1 or
// 2 CTAs per tile), SCHED (where the launch's problems and tile order come from: one
// problem, up to three in the parameter block, or a table in global memory -- the
// experts of an MoE layer) and OP (bf16 or E4M3 operands).  One CTA per SM:
//
//   warp 0      TMA producer: A/B k-blocks into a STAGES-deep shared-memory ring
//   warp 1      TMEM owner and MMA issuer: tcgen05.mma into one of two TMEM
//               accumulators (2 x 256 fp32 columns = all 512 TMEM columns), or into
//               both for one 256 x 512 tile (EPI_STORE_W)
//   warp 2      epilogue-input producer (STORE_ADD): TMA-prefetches the residual
//               tiles that the epilogue consumes
//   warp 3      idle
//   warps 4..   epilogue (4 warps; 8 for the store-only epilogues, two per quadrant):
//               TMEM -> registers (lane quadrant = warp % 4), the epilogue math,
//               tiles staged in shared memory, TMA stores
//
// CG = 1: each CTA computes a 128 x 256 output tile with cta_group::1 MMAs.
// CG = 2: a cluster of two CTAs computes a 256 x 256 tile with cta_group::2 MMAs.
//         Each CTA loads its own 128 rows of A and its own 128 rows (N) of B, both
//         CTAs' loads complete on the leader CTA's (rank 0) stage barrier, the
//         leader issues the 256 x 256 x 16 MMAs and multicasts its commits to both
//         CTAs, and each CTA drains its own 128 accumulator rows.  Per k-block a CTA
//         moves 32 KB instead of 48 KB, so the ring holds more stages and L2 serves
//         a third less.
//
// Epilogues:
//   EPI_STORE       C = acc rounded to bf16.
//   EPI_STORE_W     the same epilogue over 256 x 512 tiles (CTA pairs): both TMEM
//                   accumulators hold one tile, each A k-block feeds two N = 256 MMAs,
//                   so a k-block's operands carry 3/4 of the bytes per FLOP of a
//                   256 x 256 tile.  The accumulators form a ring of two 256-column
//                   slots: a tile takes two slots (one at a ragged N edge), the epilogue
//                   drains and returns them one at a time.
//   EPI_STORE_ADD_W EPI_STORE_ADD over 256 x 512 tiles (the residual block's grouped backward).
//   EPI_SWIGLU_FWD  B holds two W1 row slabs, [j0, j0+128) and [H+j0, H+j0+128), so
//                   accumulator columns [0,128) are `left` and [128,256) the matching
//                   `gate`.  Stores preact (both halves, bf16) and
//                   h = bf16(left * bf16(silu(gate))) computed from the bf16 preact.
//   EPI_STORE_ADD   C = bf16(acc + R) for problems flagged `res`: R [M, N] is TMA-prefetched
//                   by warp 2 like the backward's preact (the residual-add epilogue of the
//                   "Transformer MLP, GEMM and operator fusion" lesson, section 24: the down
//                   projection adds the block input; the backward's dx adds dy).
//   EPI_SWIGLU_BWD  acc = grad_h[m0:, j0:j0+256] (dy @ W2), never written out.  With the
//                   saved left/gate (each epilogue warp TMA-loads its own 32 x 64 chunks
//                   into its own slot): dleft = grad_h * silu(gate),
//                   dgate = grad_h * left * silu'(gate), silu' = sigma + silu*(1 - sigma),
//                   h = bf16(left * bf16(silu(gate))); stores grad_preact = [dleft|dgate]
//                   and h through the same slot, in 64-column tiles.
// With FP8 operands (OP_E4M3, the quantised GEMM epilogue of the lesson above, section
// 26) the epilogue first multiplies the accumulator by the operands' scale product, and
// the SwiGLU forward stores h quantised to E4M3, sat8(round(h / s_h)).
// The SwiGLU forms follow the "SwiGLU MLP Drop-H technical report" (original math,
// and the fused backward kernel's pseudo-code) and the fused dout-GEMM + SwiGLU
// backward of the "SwiGLU MLP forward/backward optimization" note (section 4): the
// activation gradient stays on chip, sigma/silu are recomputed from the saved preact.
//
// Every mbarrier wait is bounded (KernelArgs::timeout_ns, on %globaltimer); a wait
// that runs out records its role in the device error word, raises a CTA-wide abort
// flag, every role stops issuing, drains what it has in flight (again bounded),
// and the CTA frees its TMEM and returns.
#pragma once

#include <cuda_bf16.h>
#include <cstddef>
#include <cstdint>
#include <type_traits>

#include "ptx.cuh"

namespace swiglu {

enum EpiKind : int {
    EPI_STORE = 0, EPI_SWIGLU_FWD = 1, EPI_SWIGLU_BWD = 2, EPI_STORE_ADD = 3, EPI_STORE_W = 4, EPI_STORE_ADD_W = 5
};

// Operand type of the MMAs: bf16 (kind::f16) or FP8 E4M3 (kind::f8f6f4).  Both fill a
// 128-byte swizzle row per k-block -- 64 bf16 or 128 FP8 values -- so the stage
// layout, descriptors and 32-byte k-steps are the same.
enum OperandType : int { OP_BF16 = 0, OP_E4M3 = 1 };

constexpr int BM = 128;           // accumulator rows per CTA
constexpr int BN = 256;           // accumulator columns
constexpr int BK = 64;            // one 128-byte swizzle row of bf16
constexpr int UMMA_K = 16;
constexpr int NUM_THREADS = 256;
constexpr int EPI_WARP0 = 4;
constexpr int CHUNK = 32;         // epilogue columns per TMEM load
constexpr uint32_t TMEM_COLS = 512;
// The fused backward's epilogue takes the saved preact and writes its outputs in chunks
// of PRE_COLS columns: 128-byte rows, the widest a TMA box with 128-byte swizzle moves
// (each row of a box is one memory request, so wide rows mean few requests).
constexpr int PRE_COLS = 64;
constexpr int NPRE = BN / PRE_COLS;

// Device error word bits (one per role that gave up waiting).
constexpr int ERR_PRODUCER = 1, ERR_MMA = 2, ERR_EPILOGUE = 4, ERR_AUX = 8;
// Test hook: the producer issues nothing, so the consumers' waits run out.
constexpr int DEBUG_SKIP_PRODUCER = 1;

// One GEMM of a launch.  A launch runs one problem, or (EPI_STORE) up to
// MAX_PROBLEMS independent ones whose tiles share the persistent grid.
constexpr int MAX_PROBLEMS = 3;
struct Problem {
    int M;            // GEMM rows
    int N;            // EPI_STORE: GEMM columns; SWIGLU epilogues: H
    int K;
    int tiles_m;      // tiles of BM * CG rows
    int tiles_n;
    int band;         // n-tiles per raster band (L2 reuse)
    int k_blocks;
    int a_mn, b_mn;   // operand major-ness (1 = M- or N-contiguous)
    int a3d, b3d;     // an MN-major operand whose M (N) is a multiple of 64 has a 3-D map
                      // (64, K, MN / 64): one copy per k-block instead of one per 64 rows
    int res;          // EPI_STORE_ADD: add the residual tensor (tensor map i0) to this problem's output
    int tile_begin;   // index of this problem's first tile in the launch
    int no_o0;        // EPI_SWIGLU_FWD: do not store preact (o0), only h
    int slots;        // EPI_STORE_W: 256-column accumulator slots per tile (2: 256 x 512 tiles; 1: 256 x 256)
};

struct KernelArgs {
    CUtensorMap a[MAX_PROBLEMS], b[MAX_PROBLEMS], o0[MAX_PROBLEMS];
    CUtensorMap o1, i0;   // SWIGLU epilogues: h output; preact input (backward) / residual [M, N] (EPI_STORE_ADD)
    Problem prob[MAX_PROBLEMS];
    int num_problems;
    int num_tiles;
    unsigned long long timeout_ns;
    int* err;         // device error word
    int debug_flags;
    float scale_acc;  // OP_E4M3: the accumulator's scale (product of the operands' scales)
    float scale_out;  // OP_E4M3 SwiGLU forward: 1 / the scale h is quantised with
};

// A launch with an explicit per-cluster tile list (longest tiles first, balanced on
// the host): cluster c runs tiles sched[sched_off[c] .. sched_off[c + 1]).
constexpr int MAX_CLUSTERS = 128;
constexpr int MAX_SCHED = 12288;

// Split tiles (one GEMM in 256 x 512 tiles with a host list: EPI_STORE_W, or EPI_STORE_ADD_W,
// whose split tiles add the residual once, in the piece that stores the tile).  The last
// tiles of such a launch may each be shared by two CTA pairs, one summing the tile's first
// k-blocks (its prefix piece), the other the rest (its suffix piece), so that every pair
// gets the same number of k-blocks.  A list entry with SCHED_PIECE set is such a piece: its
// k-block range and split index are split[c][0] (the suffix piece of cluster c) or
// split[c][1] (with SCHED_PIECE_PREFIX).  Each epilogue warp of each piece owns one
// counter pair per accumulator slot, zero before the launch: the warp that arrives first
// writes its fp32 sums to split_sums and raises the second word; the other adds them to
// its own and stores the tile.  fp32 addition of two terms is commutative, so the result
// does not depend on which piece arrives first.
constexpr int MAX_SPLIT = 80;
constexpr int SCHED_TILE_MASK = 0x3FFF, SCHED_PIECE_PREFIX = 0x4000, SCHED_PIECE = 0x8000;
constexpr int SPLIT_WARPS = 8, SPLIT_COLS = 128;   // epilogue warps of the 256 x 512 stores; columns per warp and slot
constexpr int SPLIT_UNITS = 2 * SPLIT_WARPS * 2;  // (CTA, epilogue warp, slot) blocks of one split tile
constexpr int SPLIT_UNIT_FLOATS = 32 * SPLIT_COLS;
struct SplitPiece {
    uint16_t kb0, kb1;   // k-block range of the piece
    uint16_t id;         // split index of the tile (< MAX_SPLIT)
    uint16_t pad;
};
struct ScheduledArgs : KernelArgs {
    uint16_t sched_off[MAX_CLUSTERS + 1];
    uint16_t sched[MAX_SCHED];
    SplitPiece split[MAX_CLUSTERS][2];
    float* split_sums;   // [MAX_SPLIT][SPLIT_UNITS][SPLIT_UNIT_FLOATS]
    int* split_flags;    // [MAX_SPLIT][SPLIT_UNITS][2]: arrivals, sums written
};
static_assert(sizeof(ScheduledArgs) <= 32764, "kernel parameter block limit");
static_assert(MAX_SCHED <= SCHED_TILE_MASK + 1, "tile indices fit below the piece bits");

// Where a launch finds its problems and tile order:
//   SRC_SINGLE  one problem in the parameter block, tiles round robin over the clusters;
//   SRC_PARAMS  up to MAX_PROBLEMS problems and a host tile list in the parameter block;
//   SRC_TABLE   any number of problems (the experts of an MoE layer, each with its own
//               row count) in a table in global memory, written by the host before the
//               launch, with the host tile list beside it.  Cluster c runs the entries
//               sched[sched_off[c] .. sched_off[c + 1]), each problem << 20 | tile;
//   SRC_TABLE_COMMON  a table whose problems all share k_blocks, a_mn and b_mn (the
//               experts of one MoE GEMM): the producer takes those three from the
//               parameter block.
// The producer's mainloop issues one TMA copy per operand and k-block.  When its
// operand layout (a_mn, b_mn) comes from fixed offsets of the parameter block or is a
// compile-time constant, those copies issue at about twice the rate measured when it
// comes from a run-time-selected problem (a table entry, shared memory or a parameter
// selected by index): 15-17 % of a producer-bound GEMM.  So the list source gives the
// producer one copy of its tile body per problem index, uniform tables carry the
// layout in the parameters, and other tables get one copy per operand layout.
constexpr int SRC_SINGLE = 0, SRC_PARAMS = 1, SRC_TABLE = 2, SRC_TABLE_COMMON = 3;
__host__ __device__ constexpr bool is_table(int src) { return src >= SRC_TABLE; }
constexpr int TABLE_TILE_BITS = 20;
struct alignas(128) TableEntry {
    CUtensorMap a, b, o0;
    CUtensorMap o1, i0;   // as in KernelArgs, per problem
    Problem prob;
};
static_assert(sizeof(TableEntry) % 128 == 0 && offsetof(TableEntry, i0) % 64 == 0,
              "tensor maps in the table stay 64-byte aligned");
struct TableArgs {
    const TableEntry* table;
    const int* sched_off;
    const int* sched;
    int num_problems;
    int num_tiles;
    unsigned long long timeout_ns;
    int* err;
    int debug_flags;
    int common_k_blocks, common_a_mn, common_b_mn;   // SRC_TABLE_COMMON: shared by every problem
    int common_a3d, common_b3d;
};

template <int EPI, int CG>
struct Cfg {
    // Mainloop depth is what these kernels are most sensitive to, so the epilogue
    // buffers get what is left (single-CTA SWIGLU_FWD: 4 stages and single-buffered
    // outputs measured 11% faster than 3 / 2).  The fused backward reads its accumulator
    // 16 columns at a time (x16 TMEM loads) and moves preact and its outputs through one
    // 8 KB slot per epilogue warp, which leaves room for six operand stages (CTA pairs).
    static constexpr int CK = EPI == EPI_SWIGLU_BWD ? 16 : CHUNK;   // epilogue columns per chunk
    // 256 x 512 tiles (EPI_STORE_W): two 256-column accumulator slots per tile
    static constexpr bool WIDE = EPI == EPI_STORE_W || EPI == EPI_STORE_ADD_W;
    static constexpr bool ADD = EPI == EPI_STORE_ADD || EPI == EPI_STORE_ADD_W;   // residual-add store
    static_assert(!WIDE || CG == 2, "256 x 512 tiles are CTA-pair tiles");
    static constexpr int SLOTS = WIDE ? 2 : 1;
    static constexpr int STAGES =
        WIDE ? 4
             : CG == 1 ? ((EPI == EPI_STORE || EPI == EPI_SWIGLU_FWD || EPI == EPI_SWIGLU_BWD) ? 4 : 3)
                       : ((EPI == EPI_STORE || EPI == EPI_SWIGLU_BWD) ? 6 : 5);
    static constexpr bool STORE_ONLY = EPI == EPI_STORE || ADD || WIDE;   // one bf16 output
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_ROWS = BN / CG;                        // B rows (N) per slot held by this CTA
    static constexpr int B_SLOT_BYTES = B_ROWS * BK * 2;
    static constexpr int B_BYTES = SLOTS * B_SLOT_BYTES;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr bool BWD = EPI == EPI_SWIGLU_BWD;
    static constexpr int NOUT = (STORE_ONLY || BWD) ? 1 : 3;
    // Store-only epilogues (64 registers) run two warps per TMEM lane quadrant, each
    // draining every other chunk, so twice the TMA stores are in flight; the SwiGLU
    // epilogues need too many registers for that and keep one warp per quadrant.
    static constexpr int EPI_WARPS = STORE_ONLY ? 8 : 4;
    static constexpr int THREADS = 32 * (EPI_WARP0 + EPI_WARPS);
    // one warp's 32-row bf16 staging tile of CK columns; the fused backward's warps each own
    // one slot of two 32 x PRE_COLS tiles that first receive their preact chunk (left, gate)
    // and then stage its outputs (dleft, dgate, then h in the first tile)
    static constexpr int OUT_TILE = 32 * (BWD ? PRE_COLS : CK) * 2;
    // (single-buffered for 256 x 512 residual tiles: 4 stages of 48 KB + the residual slots
    // leave room for no more)
    static constexpr int OUT_BUFS = (EPI == EPI_STORE_ADD_W || (EPI == EPI_SWIGLU_FWD && CG == 1)) ? 1 : 2;
    static constexpr int OUT_WARP_BYTES = OUT_BUFS * NOUT * OUT_TILE;
    // epilogue-input slots of the residual (STORE_ADD): 128 rows x CK cols bf16
    static constexpr int EIN_SLOTS = ADD ? 2 : 0;
    static constexpr int EIN_SLOT_BYTES = BM * CK * 2;
    static constexpr int CHUNKS = (EPI == EPI_SWIGLU_FWD) ? (BN / 2) / CK : BN / CK;
    static constexpr int BN_PER_WARP = CHUNKS / (EPI_WARPS / 4) * CK;   // accumulator columns a warp drains per slot

    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
    static constexpr int OFF_EIN = OFF_B + STAGES * B_BYTES;
    static constexpr int OFF_OUT = OFF_EIN + EIN_SLOTS * EIN_SLOT_BYTES;
    static constexpr int OFF_BAR = OFF_OUT + EPI_WARPS * OUT_WARP_BYTES;
    // barriers: full[S], empty[S], tmem_full[2], tmem_empty[2], ein_full[E], ein_empty[E], drain,
    // and the fused backward's per-warp preact slots: slot_full[4]
    static constexpr int NUM_BARS = 2 * STAGES + 4 + 2 * EIN_SLOTS + 1 + (BWD ? 4 : 0);
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;       // tmem base, abort flag
    static constexpr int SMEM_USED = OFF_MISC + 16;
    static constexpr int SMEM_BYTES = SMEM_USED + 1024;           // slack to align the base
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

// ---------------------------------------------------------------------------
// UMMA descriptors
// ---------------------------------------------------------------------------

// Shared-memory matrix descriptor, 128-byte swizzle.
//   K-major : rows of 64 bf16 (128 B), 8-row groups 1024 B apart (SBO); LBO unused.
//   MN-major: 64 MN-contiguous elements per 128-B row, one row per k; 8-k-row groups
//             1024 B apart (SBO); 64-element MN blocks `lbo_bytes` apart (LBO).
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr, uint32_t lbo_bytes,
                                                    uint32_t sbo_bytes) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFF) >> 4);
    d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFF) << 32;
    d |= (uint64_t)1 << 46;   // descriptor version for tcgen05
    d |= (uint64_t)2 << 61;   // 128-byte swizzle
    return d;
}

// Instruction descriptor, kind::f16: bf16 A/B, fp32 D, M = 128 * CG, N = 256.
__host__ __device__ constexpr uint32_t umma_idesc(bool a_mn_major, bool b_mn_major, int cg, bool e4m3 = false) {
    return (1u << 4)                          // D format f32
           | ((e4m3 ? 0u : 1u) << 7)          // A format: bf16 (kind::f16) or E4M3 (kind::f8f6f4)
           | ((e4m3 ? 0u : 1u) << 10)         // B format likewise
           | ((a_mn_major ? 1u : 0u) << 15)   // A major-ness
           | ((b_mn_major ? 1u : 0u) << 16)   // B major-ness
           | ((uint32_t)(BN >> 3) << 17)      // N >> 3
           | ((uint32_t)((BM * cg) >> 4) << 24);   // M >> 4
}

// ---------------------------------------------------------------------------
// helpers
// ---------------------------------------------------------------------------

__device__ __forceinline__ void tile_coords(const Problem& p, int t, int& tm, int& tn) {
    const int band_tiles = p.band * p.tiles_m;
    const int b = t / band_tiles;
    const int r = t - b * band_tiles;
    const int n0 = b * p.band;
    const int w = min(p.band, p.tiles_n - n0);
    tm = r / w;
    tn = n0 + (r - tm * w);
}

// Output columns per tile of problem p: 512 for a problem of 256 x 512 tiles, else 256
// (a launch of 256 x 512 tiles may carry problems of 256 x 256 tiles beside them).
template <class C>
__device__ __forceinline__ int tile_cols(const Problem& p) {
    if constexpr (C::WIDE) return p.slots * BN;
    else return BN;
}

// Accumulator slots (256 columns each) of the tile in column-tile tn: two for a 256 x 512
// tile unless its second half lies wholly past N.
template <class C>
__device__ __forceinline__ int tile_slots(const Problem& p, int tn) {
    if constexpr (C::WIDE) return p.slots == 2 && tn * 2 * BN + BN < p.N ? 2 : 1;
    else return 1;
}

// Which problem a launch-wide tile index belongs to.
__device__ __forceinline__ int problem_of(const KernelArgs& a, int t) {
    int pi = 0;
    if (a.num_problems > 1 && t >= a.prob[1].tile_begin) pi = 1;
    if (a.num_problems > 2 && t >= a.prob[2].tile_begin) pi = 2;
    return pi;
}

// Per-problem fields selected with constant indices only: indexing the parameter
// block with a run-time value makes every access go through generic loads (and
// measured 12-20% slower mainloops).
template <class T>
__device__ __forceinline__ const T* pick3(int pi, const T* p0, const T* p1, const T* p2) {
    return pi == 0 ? p0 : (pi == 1 ? p1 : p2);
}

// The tiles of cluster c: round robin over the launch, or the host's list.
template <int SRC, class Args>
__device__ __forceinline__ int tiles_first(const Args& a, int c) {
    if constexpr (SRC != SRC_SINGLE) return a.sched_off[c];
    else return c;
}
template <int SRC, class Args>
__device__ __forceinline__ int tiles_end(const Args& a, int c) {
    if constexpr (SRC != SRC_SINGLE) return a.sched_off[c + 1];
    else return a.num_tiles;
}

// The problem of the launch's it-th tile (of this cluster's list), its index pi and
// the tile's index lt within the problem.  Returned by value: the callers' asm
// statements clobber memory, and parameter or table fields would be reloaded.
template <int SRC, class Args>
__device__ __forceinline__ Problem problem_at(const Args& a, int it, int& pi, int& lt) {
    if constexpr (is_table(SRC)) {
        const int v = __ldg(a.sched + it);
        pi = v >> TABLE_TILE_BITS;
        lt = v & ((1 << TABLE_TILE_BITS) - 1);
        return a.table[pi].prob;
    } else if constexpr (SRC == SRC_PARAMS) {
        const int t = a.sched[it] & SCHED_TILE_MASK;
        pi = problem_of(a, t);
        const Problem pr = *pick3(pi, &a.prob[0], &a.prob[1], &a.prob[2]);
        lt = t - pr.tile_begin;
        return pr;
    } else {
        pi = 0;
        lt = it;
        return a.prob[0];
    }
}

// k-block range [kb0, kb1) of the it-th entry of cluster c's list and, for a piece of a
// split tile, the tile's split index (else -1).
__device__ __forceinline__ int split_piece(const ScheduledArgs& a, int c, int it, int k_blocks, int& kb0, int& kb1) {
    const int raw = a.sched[it];
    if (!(raw & SCHED_PIECE)) {
        kb0 = 0;
        kb1 = k_blocks;
        return -1;
    }
    const SplitPiece s = a.split[c][(raw & SCHED_PIECE_PREFIX) ? 1 : 0];
    kb0 = s.kb0;
    kb1 = s.kb1;
    return s.id;
}

// Bounded wait for a flag another CTA of the launch raises (acquire).  False, with the
// role recorded and the abort flag raised, when the limit runs out.
__device__ __noinline__ bool wait_flag_bounded(const int* f, unsigned long long timeout_ns, int* err,
                                               volatile int* abort_flag, int role) {
    const uint64_t start = ptx::globaltimer();
    for (uint32_t n = 1;; ++n) {
        if (ptx::ld_acquire_gpu(f) != 0) return true;
        if ((n & 63) == 0) {
            if (*abort_flag) return false;
            if (ptx::globaltimer() - start > timeout_ns) {
                *abort_flag = 1;
                atomicOr(err, role);
                return false;
            }
        }
    }
}

enum MapId { MAP_A, MAP_B, MAP_O0, MAP_O1, MAP_I0 };
template <int SRC, int WHICH, class Args>
__device__ __forceinline__ const CUtensorMap* map_of(const Args& a, int pi) {
    if constexpr (is_table(SRC)) {
        const TableEntry* e = a.table + pi;
        if constexpr (WHICH == MAP_A) return &e->a;
        else if constexpr (WHICH == MAP_B) return &e->b;
        else if constexpr (WHICH == MAP_O0) return &e->o0;
        else if constexpr (WHICH == MAP_O1) return &e->o1;
        else return &e->i0;
    } else {
        if constexpr (WHICH == MAP_O1) return &a.o1;
        else if constexpr (WHICH == MAP_I0) return &a.i0;
        else {
            const CUtensorMap* m = WHICH == MAP_A ? a.a : (WHICH == MAP_B ? a.b : a.o0);
            if constexpr (SRC == SRC_PARAMS) return pick3(pi, &m[0], &m[1], &m[2]);
            else return &m[0];
        }
    }
}

// Bounded wait on an mbarrier phase.  Returns false (after recording `role` in the
// error word and raising the CTA abort flag) when the limit runs out, or when
// another role has already aborted.  The first probe is inline; only a wait that
// has to spin calls out.
__device__ __noinline__ bool wait_bounded_slow(uint32_t bar, uint32_t parity, unsigned long long timeout_ns,
                                               int* err, volatile int* abort_flag, int role) {
    const uint64_t start = ptx::globaltimer();
    for (uint32_t n = 1;; ++n) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if ((n & 63) == 0) {
            if (*abort_flag) return false;
            if (ptx::globaltimer() - start > timeout_ns) {
                *abort_flag = 1;
                atomicOr(err, role);
                return false;
            }
        }
    }
}

__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, unsigned long long timeout_ns, int* err,
                                             volatile int* abort_flag, int role) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    return wait_bounded_slow(bar, parity, timeout_ns, err, abort_flag, role);
}

// Short bounded wait used only while draining after an abort.
__device__ __noinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    const uint64_t start = ptx::globaltimer();
    while (!ptx::mbar_try_wait(bar, parity)) {
        if (ptx::globaltimer() - start > limit_ns) return;
    }
}

// Spin for `ns` nanoseconds (lets copies already issued land after an abort when
// their completion barrier lives in the other CTA of the pair).
__device__ __noinline__ void spin_ns(uint64_t ns) {
    const uint64_t start = ptx::globaltimer();
    while (ptx::globaltimer() - start < ns) {
    }
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }
__device__ __forceinline__ float round_bf16(float x) {
    return __bfloat162float(__float2bfloat16_rn(x));
}

// sigma(g) = 1 / (1 + e^-g) with e^-g = 2^(-g * log2 e): MUFU ex2 then MUFU rcp.
// g -> -inf: ex2 -> +inf, rcp -> 0.  g -> +inf: ex2 -> 0, sigma -> 1.
__device__ __forceinline__ float sigmoid_mufu(float g) {
    constexpr float kLog2e = 1.4426950408889634f;
    return ptx::rcp_approx(1.0f + ptx::ex2_approx(-g * kLog2e));
}

// 16-byte unit `c` (0..3) of row `r` in a [rows][64 B] tile with 64-byte swizzle.
__device__ __forceinline__ uint32_t sw64_offset(int r, int c) {
    return (uint32_t)(r * 64 + ((c ^ ((r >> 1) & 3)) << 4));
}

// 16-byte unit `c` (0..1) of row `r` in a [rows][32 B] tile with 32-byte swizzle.
__device__ __forceinline__ uint32_t sw32_offset(int r, int c) {
    return (uint32_t)(r * 32 + ((c ^ ((r >> 2) & 1)) << 4));
}

// Unit `c` of row `r` in a staging tile of CK bf16 columns (64- or 32-byte rows).
template <int CK>
__device__ __forceinline__ uint32_t stage_offset(int r, int c) {
    return CK == 32 ? sw64_offset(r, c) : sw32_offset(r, c);
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------

template <int EPI, int CG, int SCHED>
using ArgsOf = typename std::conditional<
    is_table(SCHED), TableArgs,
    typename std::conditional<SCHED == SRC_PARAMS, ScheduledArgs, KernelArgs>::type>::type;

template <int EPI, int CG, int SCHED, int OP = OP_BF16>
__global__ void __launch_bounds__(Cfg<EPI, CG>::THREADS, 1)
    gemm_kernel(const __grid_constant__ ArgsOf<EPI, CG, SCHED> args) {
    using C = Cfg<EPI, CG>;
    // pieces of split tiles: one GEMM in 256 x 512 tiles over a host list
    constexpr bool SPLIT = (EPI == EPI_STORE_W || EPI == EPI_STORE_ADD_W) && SCHED == SRC_PARAMS;
    static_assert(!SPLIT || (C::EPI_WARPS == SPLIT_WARPS && C::BN_PER_WARP == SPLIT_COLS),
                  "split-tile sums: one block of 32 rows x SPLIT_COLS per epilogue warp and slot");
    static_assert(OP == OP_BF16 || ((EPI == EPI_STORE || EPI == EPI_SWIGLU_FWD) && SCHED == SRC_SINGLE),
                  "FP8 operands: forward kernels, one problem per launch");
    constexpr int BKE = OP == OP_E4M3 ? 2 * BK : BK;   // k values per 128-byte k-block
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = ptx::smem_u32(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw_addr);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = CG == 2 ? ptx::cluster_ctarank() : 0u;   // position in the CTA pair
    const bool leader = rank == 0;
    const int cluster = blockIdx.x / CG;
    const int num_clusters = gridDim.x / CG;
    const unsigned long long tmo = args.timeout_ns;
    int* const err = args.err;
    const int t_first = tiles_first<SCHED>(args, cluster);
    const int t_end = tiles_end<SCHED>(args, cluster);
    const int t_step = SCHED ? 1 : num_clusters;

    const uint32_t bar0 = base + C::OFF_BAR;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (C::STAGES + s); };
    auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * C::STAGES + b); };
    auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * C::STAGES + 2 + b); };
    auto ein_full_bar = [&](int s) { return bar0 + 8u * (2 * C::STAGES + 4 + s); };
    auto ein_empty_bar = [&](int s) { return bar0 + 8u * (2 * C::STAGES + 4 + C::EIN_SLOTS + s); };
    const uint32_t drain_bar = bar0 + 8u * (2 * C::STAGES + 4 + 2 * C::EIN_SLOTS);
    auto slot_full_bar = [&](int w) { return drain_bar + 8u * (1 + w); };   // fused backward, epilogue warp w
    volatile uint32_t* tmem_holder = reinterpret_cast<volatile uint32_t*>(base_ptr + C::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + C::OFF_MISC + 4);

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            ptx::mbar_init(full_bar(s), 1);
            ptx::mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(tfull_bar(b), 1);
            ptx::mbar_init(tempty_bar(b), C::EPI_WARPS * CG);   // every epilogue warp of the pair
        }
        for (int s = 0; s < C::EIN_SLOTS; ++s) {
            ptx::mbar_init(ein_full_bar(s), 1);
            ptx::mbar_init(ein_empty_bar(s), 4);
        }
        ptx::mbar_init(drain_bar, 1);
        if (C::BWD)
            for (int w = 0; w < 4; ++w) ptx::mbar_init(slot_full_bar(w), 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
        if constexpr (!is_table(SCHED)) {
#pragma unroll
            for (int q = 0; q < MAX_PROBLEMS; ++q) {
                if (q < args.num_problems) {
                    ptx::prefetch_tmap(&args.a[q]);
                    ptx::prefetch_tmap(&args.b[q]);
                    if (!args.prob[q].no_o0) ptx::prefetch_tmap(&args.o0[q]);
                }
            }
            if (!C::STORE_ONLY) ptx::prefetch_tmap(&args.o1);
            if (EPI == EPI_SWIGLU_BWD || C::ADD) ptx::prefetch_tmap(&args.i0);
        }
    }
    if (warp == 1) {
        if (CG == 2) {
            ptx::tmem_alloc_pair(ptx::smem_u32((const void*)tmem_holder), TMEM_COLS);
            ptx::tmem_relinquish_pair();
        } else {
            ptx::tmem_alloc(ptx::smem_u32((const void*)tmem_holder), TMEM_COLS);
            ptx::tmem_relinquish();
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (CG == 2) ptx::cluster_sync();   // the peer's barriers exist before anything signals them
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0 && !(args.debug_flags & DEBUG_SKIP_PRODUCER)) {
            const uint32_t full_bar_leader = CG == 2 ? ptx::mapa_shared(full_bar(0), 0) : 0u;
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued = 0, last_par = 0;   // per stage: a copy was issued, and its phase parity
            bool ok = true;
            int seen_pi = -1;
            for (int it = t_first; it < t_end && ok; it += t_step) {
                int pi, lt;
                // per-tile fields in registers: the asm statements below clobber memory
                const Problem pr = problem_at<SCHED>(args, it, pi, lt);
                const CUtensorMap* mA = map_of<SCHED, MAP_A>(args, pi);
                const CUtensorMap* mB = map_of<SCHED, MAP_B>(args, pi);
                if (is_table(SCHED) && pi != seen_pi) {
                    ptx::tmap_acquire(mA);
                    ptx::tmap_acquire(mB);
                    seen_pi = pi;
                }
                // One tile's k-blocks.  Called with parameter-block fields wherever the
                // source allows it (see SRC_TABLE_COMMON).
                auto tile = [&](const Problem& p, int kb_begin, int kb_end, bool a_mn, bool b_mn, bool a3d, bool b3d,
                                const CUtensorMap* ma, const CUtensorMap* mb) {
                    int tm, tn;
                    tile_coords(p, lt, tm, tn);
                    const int m0 = tm * (BM * CG) + BM * (int)rank;   // this CTA's A rows
                    const int w = tile_slots<C>(p, tn);
                    const uint32_t tx = (uint32_t)((C::A_BYTES + w * C::B_SLOT_BYTES) * CG);
                    for (int kb = kb_begin; kb < kb_end; ++kb) {
                        if (!wait_bounded(empty_bar(stage), phase ^ 1u, tmo, err, abort_flag, ERR_PRODUCER)) {
                            ok = false;
                            break;
                        }
                        const uint32_t fb_local = full_bar(stage);
                        // CG == 2: both CTAs' copies complete on the leader's stage barrier.
                        const uint32_t fb = CG == 2 ? full_bar_leader + 8u * stage : fb_local;
                        if (leader) ptx::mbar_arrive_expect_tx(fb_local, tx);
                        issued |= 1u << stage;
                        last_par = (last_par & ~(1u << stage)) | (phase << stage);
                        const int k0 = kb * BKE;
                        const uint32_t sA = base + C::OFF_A + stage * C::A_BYTES;
                        const uint32_t sB = base + C::OFF_B + stage * C::B_BYTES;
                        auto load2 = [&](uint32_t dst, const CUtensorMap* m, int c0, int c1) {
                            if (CG == 2) ptx::tma_load_2d_pair(dst, m, fb, c0, c1);
                            else ptx::tma_load_2d(dst, m, fb, c0, c1);
                        };
                        auto load3 = [&](uint32_t dst, const CUtensorMap* m, int c1, int c2) {
                            if (CG == 2) ptx::tma_load_3d_pair(dst, m, fb, 0, c1, c2);
                            else ptx::tma_load_3d(dst, m, fb, 0, c1, c2);
                        };
                        if (a_mn) {
                            if (a3d) {
                                load3(sA, ma, k0, m0 >> 6);   // both 64-row blocks in one copy
                            } else {
                                load2(sA, ma, m0, k0);
                                load2(sA + 8192, ma, m0 + 64, k0);
                            }
                        } else {
                            load2(sA, ma, k0, m0);
                        }
                        if (EPI == EPI_SWIGLU_FWD) {
                            // W1 as (k, j, half): CG == 1 loads both slabs, CG == 2 the slab of its rank
                            const int j0 = tn * (BN / 2);
                            if (CG == 2) {
                                ptx::tma_load_3d_pair(sB, mb, fb, k0, j0, (int)rank);
                            } else {
                                ptx::tma_load_3d(sB, mb, fb, k0, j0, 0);
                                ptx::tma_load_3d(sB + C::B_BYTES / 2, mb, fb, k0, j0, 1);
                            }
                        } else {
                            // slot j of the tile: B rows [n0 + j * BN, + BN), this CTA's B_ROWS of them
                            for (int j = 0; j < w; ++j) {
                                const int n0 = tn * tile_cols<C>(p) + j * BN + C::B_ROWS * (int)rank;
                                const uint32_t sBj = sB + j * C::B_SLOT_BYTES;
                                if (!b_mn) {
                                    load2(sBj, mb, k0, n0);
                                } else if (b3d) {
                                    load3(sBj, mb, k0, n0 >> 6);   // all 64-row blocks in one copy
                                } else {
#pragma unroll
                                    for (int i = 0; i < C::B_ROWS / 64; ++i) load2(sBj + i * 8192, mb, n0 + 64 * i, k0);
                                }
                            }
                        }
                        if (++stage == C::STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                };
                if constexpr (SCHED == SRC_PARAMS) {
                    // one copy per problem index: that problem's fields at fixed offsets
                    auto fixed = [&](const Problem& p, const CUtensorMap* ma, const CUtensorMap* mb) {
                        int kb0 = 0, kb1 = p.k_blocks;
                        if constexpr (SPLIT) split_piece(args, cluster, it, p.k_blocks, kb0, kb1);
                        tile(p, kb0, kb1, p.a_mn != 0, p.b_mn != 0, p.a3d != 0, p.b3d != 0, ma, mb);
                    };
                    if (pi == 0) fixed(args.prob[0], &args.a[0], &args.b[0]);
                    else if (pi == 1) fixed(args.prob[1], &args.a[1], &args.b[1]);
                    else fixed(args.prob[2], &args.a[2], &args.b[2]);
                } else if constexpr (SCHED == SRC_TABLE_COMMON) {
                    tile(pr, 0, args.common_k_blocks, args.common_a_mn != 0, args.common_b_mn != 0, args.common_a3d != 0,
                         args.common_b3d != 0, mA, mB);
                } else if constexpr (SCHED == SRC_TABLE) {
                    // one copy per operand layout: the layout as a compile-time constant
                    const bool am = pr.a_mn != 0, bm = pr.b_mn != 0, a3 = pr.a3d != 0, b3 = pr.b3d != 0;
                    if (am && bm) tile(pr, 0, pr.k_blocks, true, true, a3, b3, mA, mB);
                    else if (am) tile(pr, 0, pr.k_blocks, true, false, a3, false, mA, mB);
                    else if (bm) tile(pr, 0, pr.k_blocks, false, true, false, b3, mA, mB);
                    else tile(pr, 0, pr.k_blocks, false, false, false, false, mA, mB);
                } else {
                    tile(pr, 0, pr.k_blocks, pr.a_mn != 0, pr.b_mn != 0, pr.a3d != 0, pr.b3d != 0, mA, mB);
                }
            }
            if (!ok) {
                // Let the loads already issued land before the CTA's shared memory goes away.
                if (leader) {
                    for (int s = 0; s < C::STAGES; ++s)
                        if ((issued >> s) & 1u) drain_wait(full_bar(s), (last_par >> s) & 1u, tmo);
                } else {
                    spin_ns(100000);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (leader CTA)
        if (lane == 0 && leader) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            uint32_t slot_seq = 0;   // accumulator slots taken so far (slot slot_seq & 1 is next)
            for (int it = t_first; it < t_end && ok; it += t_step) {
                int pi, lt;
                const Problem pq = problem_at<SCHED>(args, it, pi, lt);
                int k_blocks = pq.k_blocks;   // of this entry (a piece of a split tile: its range)
                if constexpr (SPLIT) {
                    int kb0, kb1;
                    split_piece(args, cluster, it, pq.k_blocks, kb0, kb1);
                    k_blocks = kb1 - kb0;
                }
                const bool a_mn = pq.a_mn != 0, b_mn = pq.b_mn != 0;
                const uint32_t idesc = umma_idesc(a_mn, b_mn, CG, OP == OP_E4M3);
                // Descriptors of stage 0, k = 0; a stage and a 16-k step only move the start
                // address (low 14 bits, in 16-byte units, no carry below 256 KB).
                // K-major: the next 16 k sit 32 bytes further along each 128-B row;
                // MN-major: they are the next 16 rows of 128 B.
                const uint64_t a_desc0 = a_mn ? umma_desc_sw128(base + C::OFF_A, 8192, 1024)
                                              : umma_desc_sw128(base + C::OFF_A, 16, 1024);
                const uint64_t b_desc0 = b_mn ? umma_desc_sw128(base + C::OFF_B, 8192, 1024)
                                              : umma_desc_sw128(base + C::OFF_B, 16, 1024);
                const int a_kstep = a_mn ? (2048 >> 4) : (32 >> 4);
                const int b_kstep = b_mn ? (2048 >> 4) : (32 >> 4);
                int w = 1;
                if constexpr (C::WIDE) {
                    int tm, tn;
                    tile_coords(pq, lt, tm, tn);
                    w = tile_slots<C>(pq, tn);
                }
                // the tile's slots, drained by the epilogue (use u of slot b: its (u+1)-th tile)
                for (int j = 0; j < w && ok; ++j) {
                    const uint32_t s = slot_seq + (uint32_t)j;
                    if (!wait_bounded(tempty_bar(s & 1u), ((s >> 1) & 1u) ^ 1u, tmo, err, abort_flag, ERR_MMA))
                        ok = false;
                }
                if (!ok) break;
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem_base + (slot_seq & 1u) * BN;           // slot 0 of the tile
                const uint32_t d_tmem1 = tmem_base + ((slot_seq + 1u) & 1u) * BN;   // slot 1 (wide tiles)
                for (int kb = 0; kb < k_blocks; ++kb) {
                    if (!wait_bounded(full_bar(stage), phase, tmo, err, abort_flag, ERR_MMA)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint64_t ad0 = a_desc0 + (uint64_t)(stage * (C::A_BYTES >> 4));
                    const uint64_t bd0 = b_desc0 + (uint64_t)(stage * (C::B_BYTES >> 4));
#pragma unroll
                    for (int k = 0; k < BK / UMMA_K; ++k) {
                        const uint64_t ad = ad0 + (uint64_t)(k * a_kstep);
                        const uint64_t bd = bd0 + (uint64_t)(k * b_kstep);
                        const uint32_t acc_flag = (kb | k) != 0 ? 1u : 0u;
                        if (OP == OP_E4M3) {
                            if (CG == 2) ptx::mma_e4m3_pair(d_tmem, ad, bd, idesc, acc_flag);
                            else ptx::mma_e4m3(d_tmem, ad, bd, idesc, acc_flag);
                        } else {
                            if (CG == 2) ptx::mma_bf16_pair(d_tmem, ad, bd, idesc, acc_flag);
                            else ptx::mma_bf16(d_tmem, ad, bd, idesc, acc_flag);
                            if (C::WIDE && w == 2)   // the same A k-step against the second B slot
                                ptx::mma_bf16_pair(d_tmem1, ad, bd + (uint64_t)(C::B_SLOT_BYTES >> 4), idesc,
                                                   acc_flag);
                        }
                    }
                    if (CG == 2) ptx::mma_commit_pair_mc(empty_bar(stage), 0x3);
                    else ptx::mma_commit(empty_bar(stage));
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                for (int j = 0; j < w; ++j) {
                    const uint32_t b = (slot_seq + (uint32_t)j) & 1u;
                    if (CG == 2) ptx::mma_commit_pair_mc(tfull_bar(b), 0x3);
                    else ptx::mma_commit(tfull_bar(b));
                }
                slot_seq += (uint32_t)w;
            }
            if (!ok) {
                if (CG == 2) ptx::mma_commit_pair_mc(drain_bar, 0x1);
                else ptx::mma_commit(drain_bar);
                drain_wait(drain_bar, 0, tmo);
            }
        }
        __syncwarp();
    } else if (warp == 2) {
        // ------------------------------------------------------------ epilogue-input producer
        if (C::ADD && lane == 0) {
            // the residual [M, N] tiles of the problems that carry one, 128 rows x 32 columns
            // per chunk, slot by slot, in the order the epilogue warps consume them
            int slot = 0;
            uint32_t phase = 0;
            int last_parity[C::EIN_SLOTS > 0 ? C::EIN_SLOTS : 1];
            for (int s = 0; s < C::EIN_SLOTS; ++s) last_parity[s] = -1;
            bool ok = true;
            int seen_pi = -1;
            for (int it = t_first; it < t_end && ok; it += t_step) {
                int pi, lt;
                const Problem pr = problem_at<SCHED>(args, it, pi, lt);
                if (!pr.res) continue;
                const CUtensorMap* mI = map_of<SCHED, MAP_I0>(args, pi);
                if (is_table(SCHED) && pi != seen_pi) {
                    ptx::tmap_acquire(mI);
                    seen_pi = pi;
                }
                int tm, tn;
                tile_coords(pr, lt, tm, tn);
                const int m0 = tm * (BM * CG) + BM * (int)rank;
                const int w = tile_slots<C>(pr, tn);
                for (int j = 0; j < w && ok; ++j) {
                    const int n0 = tn * tile_cols<C>(pr) + j * BN;
                    for (int c = 0; c < C::CHUNKS; ++c) {
                        if (!wait_bounded(ein_empty_bar(slot), phase ^ 1u, tmo, err, abort_flag, ERR_AUX)) {
                            ok = false;
                            break;
                        }
                        const uint32_t fb = ein_full_bar(slot);
                        ptx::mbar_arrive_expect_tx(fb, C::EIN_SLOT_BYTES);
                        last_parity[slot] = (int)phase;
                        ptx::tma_load_2d(base + C::OFF_EIN + slot * C::EIN_SLOT_BYTES, mI, fb, n0 + c * CHUNK, m0);
                        if (++slot == C::EIN_SLOTS) {
                            slot = 0;
                            phase ^= 1u;
                        }
                    }
                }
            }
            if (!ok) {
                for (int s = 0; s < C::EIN_SLOTS; ++s)
                    if (last_parity[s] >= 0) drain_wait(ein_full_bar(s), (uint32_t)last_parity[s], tmo);
            }
        }
        __syncwarp();
    } else if (warp >= EPI_WARP0 && C::BWD) {
        // ------------------------------------------------------------ fused backward epilogue
        // Each warp drains its 32 accumulator rows in chunks of PRE_COLS columns through its
        // own slot of shared memory: lane 0 TMA-loads the chunk's saved preact (left into
        // the first tile, gate into the second, 128-byte rows); every lane copies its row to
        // registers; the warp computes dleft, dgate and h from the accumulator, writes dleft
        // and dgate over the preact it no longer needs and stores them, then h into the
        // first tile once dleft's store has read it; once h's store has read the slot, the
        // next chunk's preact is loaded into it (the next tile's first chunk after the last).
        const int wq = warp & 3;                 // TMEM lane quadrant = tile rows [32wq, 32wq+32)
        const int wi = warp - EPI_WARP0;
        const uint32_t slot = base + C::OFF_OUT + wi * C::OUT_WARP_BYTES;
        const uint32_t slot_g = slot + C::OUT_TILE;
        const uint32_t sbar = slot_full_bar(wi);
        const uint32_t srow = (uint32_t)lane * 128u;   // this lane's row in a slot tile
        uint32_t spar = 0;         // parity of the slot barrier's next phase
        bool pending = false;      // a preact load is in flight into the slot
        auto load_chunk = [&](const CUtensorMap* mI, int j, int mrow) {
            if (lane == 0) {
                ptx::mbar_arrive_expect_tx(sbar, 2 * C::OUT_TILE);
                ptx::tma_load_3d(slot, mI, sbar, j, 0, mrow);     // left
                ptx::tma_load_3d(slot_g, mI, sbar, j, 1, mrow);   // gate
            }
            pending = true;
        };
        int local = 0;
        bool ok = true;
        int seen_pi = -1;
        for (int it = t_first; it < t_end && ok; it += t_step, ++local) {
            int pi, lt;
            const Problem pr = problem_at<SCHED>(args, it, pi, lt);
            const CUtensorMap* mO0 = map_of<SCHED, MAP_O0>(args, pi);
            const CUtensorMap* mO1 = map_of<SCHED, MAP_O1>(args, pi);
            const CUtensorMap* mI = map_of<SCHED, MAP_I0>(args, pi);
            if (is_table(SCHED) && pi != seen_pi && lane == 0) {
                ptx::tmap_acquire(mO0);
                ptx::tmap_acquire(mO1);
                ptx::tmap_acquire(mI);
            }
            seen_pi = pi;
            int tm, tn;
            tile_coords(pr, lt, tm, tn);
            const int mrow0 = tm * (BM * CG) + BM * (int)rank + 32 * wq;   // first row of this warp
            const bool rows_live = mrow0 < pr.M;
            if (!pending) load_chunk(mI, tn * BN, mrow0);   // (later tiles: loaded during the last)
            const int ab = local & 1;
            const uint32_t use = (uint32_t)(local >> 1);
            const bool got = __all_sync(0xffffffffu, wait_bounded(tfull_bar(ab), use & 1u, tmo, err, abort_flag,
                                                                  ERR_EPILOGUE));
            if (!got) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            const uint32_t t_row = tmem_base + ((uint32_t)(32 * wq) << 16) + (uint32_t)(ab * BN);
            for (int q = 0; q < NPRE; ++q) {
                const bool in_ok = __all_sync(0xffffffffu, wait_bounded(sbar, spar, tmo, err, abort_flag, ERR_EPILOGUE));
                if (!in_ok) {
                    ok = false;
                    break;
                }
                spar ^= 1u;
                pending = false;
                // this row's 64 left and 64 gate values (128-byte swizzle)
                uint32_t lft[32], gte[32];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const uint32_t off = srow + (uint32_t)((u ^ (lane & 7)) << 4);
                    const uint4 l4 = ptx::lds128(slot + off);
                    const uint4 g4 = ptx::lds128(slot_g + off);
                    lft[4 * u + 0] = l4.x; lft[4 * u + 1] = l4.y; lft[4 * u + 2] = l4.z; lft[4 * u + 3] = l4.w;
                    gte[4 * u + 0] = g4.x; gte[4 * u + 1] = g4.y; gte[4 * u + 2] = g4.z; gte[4 * u + 3] = g4.w;
                }
                uint32_t hb[32];   // h of the chunk, packed bf16 pairs, staged after dleft's store
#pragma unroll
                for (int i = 0; i < PRE_COLS / C::CK; ++i) {
                    uint32_t acc[16];
                    ptx::tmem_ld_32x32b_x16(t_row + q * PRE_COLS + i * C::CK, acc);
                    ptx::tmem_ld_wait();
                    if (q == NPRE - 1 && i == PRE_COLS / C::CK - 1) {
                        // accumulator fully read: hand it back to the MMA warp (of the leader CTA)
                        ptx::tc_fence_before();
                        __syncwarp();
                        if (lane == 0) {
                            if (CG == 2) ptx::mbar_arrive_cluster(ptx::mapa_shared(tempty_bar(ab), 0));
                            else ptx::mbar_arrive(tempty_bar(ab));
                        }
                    }
                    uint32_t dl[8], dg[8];
#pragma unroll
                    for (int w = 0; w < 8; ++w) {
                        const uint32_t lw = lft[8 * i + w], gw = gte[8 * i + w];
                        float dlv[2], dgv[2], hv[2];
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const float gh = __uint_as_float(acc[2 * w + e]);
                            const float l = e ? bf16_hi(lw) : bf16_lo(lw);
                            const float g = e ? bf16_hi(gw) : bf16_lo(gw);
                            const float sig = sigmoid_mufu(g);
                            const float silu = g * sig;
                            const float silu_p = sig + silu * (1.0f - sig);
                            dlv[e] = gh * silu;
                            dgv[e] = gh * l * silu_p;
                            hv[e] = l * round_bf16(silu);
                        }
                        dl[w] = pack_bf16(dlv[0], dlv[1]);
                        dg[w] = pack_bf16(dgv[0], dgv[1]);
                        hb[8 * i + w] = pack_bf16(hv[0], hv[1]);
                    }
                    // dleft and dgate over this lane's own (already copied) preact row
                    const uint32_t u0 = srow + (uint32_t)(((2 * i) ^ (lane & 7)) << 4);
                    const uint32_t u1 = srow + (uint32_t)(((2 * i + 1) ^ (lane & 7)) << 4);
                    ptx::sts128(slot + u0, make_uint4(dl[0], dl[1], dl[2], dl[3]));
                    ptx::sts128(slot + u1, make_uint4(dl[4], dl[5], dl[6], dl[7]));
                    ptx::sts128(slot_g + u0, make_uint4(dg[0], dg[1], dg[2], dg[3]));
                    ptx::sts128(slot_g + u1, make_uint4(dg[4], dg[5], dg[6], dg[7]));
                }
                const int j = tn * BN + q * PRE_COLS;
                const bool live = rows_live && j < pr.N;
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    if (live) ptx::tma_store_3d(mO0, slot, j, 0, mrow0);     // dleft
                    ptx::bulk_commit_group();
                    if (live) ptx::tma_store_3d(mO0, slot_g, j, 1, mrow0);   // dgate
                    ptx::bulk_commit_group();
                    ptx::bulk_wait_group_read<1>();                         // dleft's tile read
                }
                __syncwarp();
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    ptx::sts128(slot + srow + (uint32_t)((u ^ (lane & 7)) << 4),
                                make_uint4(hb[4 * u], hb[4 * u + 1], hb[4 * u + 2], hb[4 * u + 3]));
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    if (live) ptx::tma_store_2d(mO1, slot, j, mrow0);        // h
                    ptx::bulk_commit_group();
                    ptx::bulk_wait_group_read<0>();                         // the slot is free
                }
                __syncwarp();
                // the next chunk's preact into the slot: this tile's next, or the next tile's first
                if (q + 1 < NPRE) {
                    load_chunk(mI, j + PRE_COLS, mrow0);
                } else if (it + t_step < t_end) {
                    int pn, ln, tmn, tnn;
                    const Problem pnx = problem_at<SCHED>(args, it + t_step, pn, ln);
                    tile_coords(pnx, ln, tmn, tnn);
                    const CUtensorMap* mIn = map_of<SCHED, MAP_I0>(args, pn);
                    if (is_table(SCHED) && pn != seen_pi && lane == 0) ptx::tmap_acquire(mIn);
                    load_chunk(mIn, tnn * BN, tmn * (BM * CG) + BM * (int)rank + 32 * wq);
                }
            }
        }
        // let a preact load still in flight land before the shared memory goes away
        if (pending) drain_wait(sbar, spar, tmo);
        if (lane == 0) ptx::bulk_wait_group<0>();
        ptx::tc_fence_before();
        __syncwarp();
    } else if (warp >= EPI_WARP0) {
        // ------------------------------------------------------------ epilogue
        const int wq = warp & 3;                 // TMEM lane quadrant = tile rows [32wq, 32wq+32)
        const int row = 32 * wq + lane;          // row within this CTA's 128 rows
        const int grp = (warp - EPI_WARP0) >> 2; // which of the quadrant's warps (store-only: 0 or 1)
        constexpr int GROUPS = C::EPI_WARPS / 4;
        const uint32_t out_base = base + C::OFF_OUT + (warp - EPI_WARP0) * C::OUT_WARP_BYTES;
        int res_slots = 0;   // residual-add stores: accumulator slots of residual problems drained so far
        int ob = 0;
        uint32_t slot_seq = 0;   // accumulator slots drained so far
        bool ok = true;
        int seen_pi = -1;
        for (int it = t_first; it < t_end && ok; it += t_step) {
            int pi, lt;
            // registers (asm statements clobber memory)
            const Problem pr = problem_at<SCHED>(args, it, pi, lt);
            const int n_limit = pr.N;
            int sid = -1;   // split index of the tile when this entry is a piece of one
            if constexpr (SPLIT) {
                int kb0, kb1;
                sid = split_piece(args, cluster, it, pr.k_blocks, kb0, kb1);
            }
            (void)sid;
            const CUtensorMap* mO0 = map_of<SCHED, MAP_O0>(args, pi);
            const CUtensorMap* mO1 = map_of<SCHED, MAP_O1>(args, pi);
            if (is_table(SCHED) && pi != seen_pi && lane == 0) {
                ptx::tmap_acquire(mO0);
                if (!C::STORE_ONLY) ptx::tmap_acquire(mO1);
            }
            seen_pi = pi;
            int tm, tn;
            tile_coords(pr, lt, tm, tn);
            const int m0 = tm * (BM * CG) + BM * (int)rank;
            const int mrow0 = m0 + 32 * wq;     // first output row of this warp's slice
            const bool rows_live = mrow0 < pr.M;
            // the tile's accumulator slots, in the order the MMA warp filled them
            const int w = tile_slots<C>(pr, tn);
            for (int sl = 0; sl < w && ok; ++sl) {
                const uint32_t s = slot_seq + (uint32_t)sl;
                const int ab = (int)(s & 1u);
                const uint32_t use = s >> 1;
                // every lane observes the barrier itself (acquire), the warp agrees on the outcome
                const bool got = __all_sync(0xffffffffu, wait_bounded(tfull_bar(ab), use & 1u, tmo, err, abort_flag,
                                                                      ERR_EPILOGUE));
                if (!got) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t t_row = tmem_base + ((uint32_t)(32 * wq) << 16) + (uint32_t)(ab * BN);

                // piece of a split tile: 1 = arrived first, writes its fp32 sums; 2 = adds them
                int split_role = 0;
                float4* sums = nullptr;
                int* sflags = nullptr;
                if constexpr (SPLIT) {
                    if (sid >= 0) {
                        const int unit = ((sid * 2 + (int)rank) * SPLIT_WARPS + (warp - EPI_WARP0)) * 2 + sl;
                        sflags = args.split_flags + 2 * unit;
                        sums = reinterpret_cast<float4*>(args.split_sums) + (size_t)unit * (SPLIT_UNIT_FLOATS / 4);
                        int old = 0;
                        if (lane == 0) old = atomicAdd(sflags, 1);
                        split_role = __shfl_sync(0xffffffffu, old, 0) == 0 ? 1 : 2;
                        if (split_role == 2) {
                            // the other piece arrived first and is writing its sums
                            int ready = 1;
                            if (lane == 0)
                                ready = wait_flag_bounded(sflags + 1, tmo, err, abort_flag, ERR_EPILOGUE) ? 1 : 0;
                            if (!__shfl_sync(0xffffffffu, ready, 0)) {
                                ok = false;
                                break;
                            }
                            __threadfence();
                        }
                    }
                }
                (void)sums;
                (void)sflags;

                constexpr bool FAST = (EPI == EPI_STORE || EPI == EPI_STORE_W || EPI == EPI_STORE_ADD_W) && OP == OP_BF16;
                if (FAST && !(C::ADD && pr.res)) {
                    // Plain bf16 stores: all of this warp's chunks of the slot into registers as
                    // packed bf16 first, then the slot goes back to the MMA warp, then the
                    // stores.  A 256 x 512 tile's next mainloop waits for its slots' release.
                    constexpr int NCH = C::CHUNKS / GROUPS;
                    uint32_t pk[NCH][16];
#pragma unroll
                    for (int i = 0; i < NCH; ++i) {
                        uint32_t acc[32];
                        ptx::tmem_ld_32x32b_x32(t_row + (grp + i * GROUPS) * CHUNK, acc);
                        ptx::tmem_ld_wait();
                        if constexpr (SPLIT) {
                            // sums as [chunk][16-byte group][lane]: each store covers 512 contiguous bytes
                            if (split_role == 1) {
#pragma unroll
                                for (int q = 0; q < 8; ++q)
                                    __stcg(sums + (i * 8 + q) * 32 + lane,
                                           make_float4(__uint_as_float(acc[4 * q]), __uint_as_float(acc[4 * q + 1]),
                                                       __uint_as_float(acc[4 * q + 2]), __uint_as_float(acc[4 * q + 3])));
                                continue;
                            }
                            if (split_role == 2) {
#pragma unroll
                                for (int q = 0; q < 8; ++q) {
                                    const float4 v = __ldcg(sums + (i * 8 + q) * 32 + lane);
                                    acc[4 * q] = __float_as_uint(__uint_as_float(acc[4 * q]) + v.x);
                                    acc[4 * q + 1] = __float_as_uint(__uint_as_float(acc[4 * q + 1]) + v.y);
                                    acc[4 * q + 2] = __float_as_uint(__uint_as_float(acc[4 * q + 2]) + v.z);
                                    acc[4 * q + 3] = __float_as_uint(__uint_as_float(acc[4 * q + 3]) + v.w);
                                }
                            }
                        }
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            pk[i][j] = pack_bf16(__uint_as_float(acc[2 * j]), __uint_as_float(acc[2 * j + 1]));
                    }
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        if (CG == 2) ptx::mbar_arrive_cluster(ptx::mapa_shared(tempty_bar(ab), 0));
                        else ptx::mbar_arrive(tempty_bar(ab));
                    }
                    if constexpr (SPLIT) {
                        if (split_role == 1) {
                            // sums written: release them to the other piece, which stores the tile
                            __threadfence();
                            __syncwarp();
                            if (lane == 0) ptx::st_release_gpu(sflags + 1, 1);
                            continue;
                        }
                    }
#pragma unroll
                    for (int i = 0; i < NCH; ++i) {
                        const int c = grp + i * GROUPS;
                        if (lane == 0) ptx::bulk_wait_group_read<C::OUT_BUFS - 1>();
                        __syncwarp();
                        const uint32_t ob_base = out_base + ob * (C::NOUT * C::OUT_TILE);
#pragma unroll
                        for (int q = 0; q < C::CK / 8; ++q)
                            ptx::sts128(ob_base + stage_offset<C::CK>(lane, q),
                                        make_uint4(pk[i][4 * q], pk[i][4 * q + 1], pk[i][4 * q + 2], pk[i][4 * q + 3]));
                        ptx::fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0 && rows_live) {
                            const int n = tn * tile_cols<C>(pr) + sl * BN + c * CHUNK;
                            if (n < n_limit) ptx::tma_store_2d(mO0, ob_base, n, mrow0);
                        }
                        if (lane == 0) ptx::bulk_commit_group();
                        ob = (ob + 1) % C::OUT_BUFS;
                    }
                } else {
                for (int c = grp; c < C::CHUNKS; c += GROUPS) {
                    uint32_t acc[32];
                    uint32_t acc2[32];
                    if (EPI == EPI_SWIGLU_FWD) {
                        ptx::tmem_ld_32x32b_x32(t_row + c * CHUNK, acc);
                        ptx::tmem_ld_32x32b_x32(t_row + BN / 2 + c * CHUNK, acc2);
                    } else {
                        ptx::tmem_ld_32x32b_x32(t_row + c * CHUNK, acc);
                    }
                    ptx::tmem_ld_wait();
                    if (c + GROUPS >= C::CHUNKS) {   // this warp's last chunk of the slot
                        // Accumulator fully read: hand it back to the MMA warp (of the leader CTA).
                        ptx::tc_fence_before();
                        __syncwarp();
                        if (lane == 0) {
                            if (CG == 2) ptx::mbar_arrive_cluster(ptx::mapa_shared(tempty_bar(ab), 0));
                            else ptx::mbar_arrive(tempty_bar(ab));
                        }
                    }
                    if constexpr (SPLIT) {
                        // a piece of a split tile (residual store): the sums as in the plain store
                        const int i = (c - grp) / GROUPS;
                        if (split_role == 1) {
#pragma unroll
                            for (int q = 0; q < 8; ++q)
                                __stcg(sums + (i * 8 + q) * 32 + lane,
                                       make_float4(__uint_as_float(acc[4 * q]), __uint_as_float(acc[4 * q + 1]),
                                                   __uint_as_float(acc[4 * q + 2]), __uint_as_float(acc[4 * q + 3])));
                        } else if (split_role == 2) {
#pragma unroll
                            for (int q = 0; q < 8; ++q) {
                                const float4 v = __ldcg(sums + (i * 8 + q) * 32 + lane);
                                acc[4 * q] = __float_as_uint(__uint_as_float(acc[4 * q]) + v.x);
                                acc[4 * q + 1] = __float_as_uint(__uint_as_float(acc[4 * q + 1]) + v.y);
                                acc[4 * q + 2] = __float_as_uint(__uint_as_float(acc[4 * q + 2]) + v.z);
                                acc[4 * q + 3] = __float_as_uint(__uint_as_float(acc[4 * q + 3]) + v.w);
                            }
                        }
                    }

                    // epilogue input of the residual store: the residual's 32 columns
                    uint32_t lft[16];
                    if (C::ADD && pr.res) {
                        constexpr int NSLOT = C::EIN_SLOTS > 0 ? C::EIN_SLOTS : 1;
                        const int q = res_slots * C::CHUNKS + c;
                        const int slot = q % NSLOT;
                        const bool in_ok = __all_sync(0xffffffffu, wait_bounded(ein_full_bar(slot),
                                                                                (uint32_t)((q / NSLOT) & 1), tmo,
                                                                                err, abort_flag, ERR_EPILOGUE));
                        if (!in_ok) {
                            ok = false;
                            break;
                        }
                        const uint32_t slot_base = base + C::OFF_EIN + slot * C::EIN_SLOT_BYTES;
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            const uint4 r4 = ptx::lds128(slot_base + sw64_offset(row, q4));
                            lft[4 * q4 + 0] = r4.x; lft[4 * q4 + 1] = r4.y; lft[4 * q4 + 2] = r4.z; lft[4 * q4 + 3] = r4.w;
                        }
                        __syncwarp();
                        if (lane == 0) ptx::mbar_arrive(ein_empty_bar(slot));
                    }
                    // the first piece of a split tile takes its residual chunk off the ring and
                    // leaves the tile to the other piece
                    if (SPLIT && split_role == 1) continue;
                    // outputs for this chunk, packed bf16 pairs (the FP8 forward's h: 4 codes a word)
                    uint32_t o0[16], o1[16], o2[16];
                    if (OP == OP_E4M3) {
                        // FP8 operands: the accumulator carries the product of the operands' scales
                        float sa = 1.0f;
                        if constexpr (OP == OP_E4M3) sa = args.scale_acc;
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            acc[i] = __float_as_uint(__uint_as_float(acc[i]) * sa);
                            if (EPI == EPI_SWIGLU_FWD) acc2[i] = __float_as_uint(__uint_as_float(acc2[i]) * sa);
                        }
                    }
                    if (EPI == EPI_STORE || EPI == EPI_STORE_W || (C::ADD && !pr.res)) {
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            o0[i] = pack_bf16(__uint_as_float(acc[2 * i]), __uint_as_float(acc[2 * i + 1]));
                    } else if (C::ADD) {
                        // residual add: C = acc + R, summed in fp32 and rounded once
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            o0[i] = pack_bf16(__uint_as_float(acc[2 * i]) + bf16_lo(lft[i]),
                                              __uint_as_float(acc[2 * i + 1]) + bf16_hi(lft[i]));
                    } else if (EPI == EPI_SWIGLU_FWD) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const uint32_t lb = pack_bf16(__uint_as_float(acc[2 * i]), __uint_as_float(acc[2 * i + 1]));
                            const uint32_t gb = pack_bf16(__uint_as_float(acc2[2 * i]), __uint_as_float(acc2[2 * i + 1]));
                            o0[i] = lb;
                            o1[i] = gb;
                            float hv[2];
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                const float l = e ? bf16_hi(lb) : bf16_lo(lb);
                                const float g = e ? bf16_hi(gb) : bf16_lo(gb);
                                const float silu = g * sigmoid_mufu(g);
                                hv[e] = l * round_bf16(silu);
                            }
                            if (OP == OP_E4M3) {
                                // the quantising epilogue: h8 = sat8(round(h / s_h)), two codes per 16 bits
                                float so = 1.0f;
                                if constexpr (OP == OP_E4M3) so = args.scale_out;
                                const uint32_t q2 = ptx::cvt_e4m3x2(hv[0] * so, hv[1] * so);
                                o2[i >> 1] = (i & 1) ? (o2[i >> 1] | (q2 << 16)) : q2;
                            } else {
                                o2[i] = pack_bf16(hv[0], hv[1]);
                            }
                        }
                    }

                    // stage in shared memory (64-byte swizzle) and TMA-store this warp's 32x32 tiles
                    if (lane == 0) ptx::bulk_wait_group_read<C::OUT_BUFS - 1>();
                    __syncwarp();
                    const uint32_t ob_base = out_base + ob * (C::NOUT * C::OUT_TILE);
#pragma unroll
                    for (int o = 0; o < C::NOUT; ++o) {
                        const uint32_t* src = (o == 0) ? o0 : (o == 1) ? o1 : o2;
                        const uint32_t tile = ob_base + o * C::OUT_TILE;
                        if (OP == OP_E4M3 && o == 2) {
                            // the FP8 h tile: 32 rows of 32 bytes, unswizzled
                            ptx::sts128(tile + lane * 32, make_uint4(src[0], src[1], src[2], src[3]));
                            ptx::sts128(tile + lane * 32 + 16, make_uint4(src[4], src[5], src[6], src[7]));
                            continue;
                        }
#pragma unroll
                        for (int q = 0; q < C::CK / 8; ++q)
                            ptx::sts128(tile + stage_offset<C::CK>(lane, q),
                                        make_uint4(src[4 * q], src[4 * q + 1], src[4 * q + 2], src[4 * q + 3]));
                    }
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0 && rows_live) {
                        if (C::STORE_ONLY) {
                            const int n = tn * tile_cols<C>(pr) + sl * BN + c * CHUNK;
                            if (n < n_limit) ptx::tma_store_2d(mO0, ob_base, n, mrow0);
                        } else {
                            const int jw = (EPI == EPI_SWIGLU_FWD) ? BN / 2 : BN;
                            const int j = tn * jw + c * C::CK;
                            if (j < n_limit) {
                                if (!pr.no_o0) {
                                    ptx::tma_store_3d(mO0, ob_base, j, 0, mrow0);
                                    ptx::tma_store_3d(mO0, ob_base + C::OUT_TILE, j, 1, mrow0);
                                }
                                ptx::tma_store_2d(mO1, ob_base + 2 * C::OUT_TILE, j, mrow0);
                            }
                        }
                    }
                    if (lane == 0) ptx::bulk_commit_group();
                    ob = (ob + 1) % C::OUT_BUFS;
                }
                }
                if constexpr (SPLIT) {
                    if (split_role == 1) {
                        // sums written: release them to the other piece
                        __threadfence();
                        __syncwarp();
                        if (lane == 0) ptx::st_release_gpu(sflags + 1, 1);
                    }
                }
                if (C::ADD && pr.res) ++res_slots;
            }
            slot_seq += (uint32_t)w;

        }
        if (lane == 0) ptx::bulk_wait_group<0>();
        ptx::tc_fence_before();
        __syncwarp();
    }

    __syncthreads();
    if (CG == 2) ptx::cluster_sync();   // no CTA leaves while its peer may still touch it
    if (warp == 1) {
        ptx::tc_fence_after();
        if (CG == 2) ptx::tmem_dealloc_pair(tmem_base, TMEM_COLS);
        else ptx::tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

}  // namespace swiglu
