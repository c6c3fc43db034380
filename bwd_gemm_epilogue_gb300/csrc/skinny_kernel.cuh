// skinny_kernel.cuh -- the block's weight-streaming products for a few tokens
// (M <= 64, the decode regime), and the element-wise kernels that finish them.
//
// With M tokens the big GEMMs degenerate: the weights are read once and used M
// times, so the work is bound by HBM bandwidth, and a 128-token tile would leave
// most SMs idle.  The products are computed transposed ("swap-AB"):
//
//   C^T [N, M] += W [N, K-slice] * X [M, K-slice]^T
//
// with the weight W as the 128-row tcgen05 A operand (K-major, or MN-major when W
// is stored transposed) and the tokens X as an N = 16..64 B operand.  The K range is
// split so that (N / 128) x splits work units cover the SMs; work unit (tile, split)
// stores its 128 x M fp32 partial into plane `split` of an fp32 buffer [splits][N][ld]
// with a TMA store.  The element-wise kernels add the planes in a fixed order, so the
// results are the same bits on every run (no order-dependent reduction).
// Element-wise kernels then round and transpose the fp32 sums into the bf16 outputs
// and apply the SwiGLU forward or backward -- for M tokens grad_h is M x H fp32
// (0.7 MB at decode sizes), so it is written once to global memory and read once
// by the SwiGLU-backward kernel instead of being consumed on chip.
//
// Warp roles as in gemm_kernel.cuh: warp 0 TMA producer, warp 1 TMEM owner and MMA
// issuer (two accumulators of <= 64 fp32 columns), warps 4..7 drain TMEM, stage the
// fp32 tile in shared memory and issue the stores.  Every wait is bounded.
#pragma once

#include "gemm_kernel.cuh"

namespace swiglu {

constexpr int SK_MAX_M = 64;            // tokens handled by this path
constexpr int SK_STAGES = 8;
constexpr int SK_A_BYTES = BM * BK * 2;                 // 128 weight rows x 64 k
constexpr int SK_B_BYTES = SK_MAX_M * BK * 2;           // <= 64 token rows x 64 k
constexpr int SK_STAGE_BYTES = SK_A_BYTES + SK_B_BYTES;
constexpr int SK_OUT_WARP = 32 * SK_MAX_M * 4;          // 32 rows x 64 fp32
constexpr int SK_OFF_B = SK_STAGES * SK_A_BYTES;
constexpr int SK_OFF_OUT = SK_OFF_B + SK_STAGES * SK_B_BYTES;
constexpr int SK_OFF_BAR = SK_OFF_OUT + 4 * SK_OUT_WARP;
constexpr int SK_NUM_BARS = 2 * SK_STAGES + 4 + 1;
constexpr int SK_OFF_MISC = SK_OFF_BAR + SK_NUM_BARS * 8;
constexpr int SK_SMEM_BYTES = SK_OFF_MISC + 16 + 1024;
static_assert(SK_SMEM_BYTES <= 232448, "shared memory budget");
constexpr uint32_t SK_TMEM_COLS = 128;                  // 2 x 64 fp32 columns

struct SkinnyArgs {
    CUtensorMap w;      // weight (MMA A): K-major box 64 x 128, or MN-major box 64 x 64 (two per stage)
    CUtensorMap x;      // tokens (MMA B) [M, K]: K-major box 64 x n_mma
    CUtensorMap out;    // fp32 partial planes (m, n, split) of [splits][N][n_mma]: box 16 x 32 x 1, 64-byte swizzle
    int N, K;
    int n_mma;          // tokens rounded up to a multiple of 16 (MMA N)
    int w_mn;           // weight stored [K, N] (N contiguous)
    int n_tiles, splits, kb_per_split, k_blocks;
    unsigned long long timeout_ns;
    int* err;
    int debug_flags;
};

// OP: bf16 operands (kind::f16) or FP8 E4M3 operands (kind::f8f6f4, 128 k values per
// 128-byte k-block; K-major weights only).  The fp32 sums are unscaled.
template <int OP = OP_BF16>
__global__ void __launch_bounds__(NUM_THREADS, 1) skinny_gemm_kernel(const __grid_constant__ SkinnyArgs args) {
    constexpr int BKE = OP == OP_E4M3 ? 2 * BK : BK;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = ptx::smem_u32(smem_raw);
    const uint32_t base = (raw_addr + 1023u) & ~1023u;
    uint8_t* base_ptr = smem_raw + (base - raw_addr);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const unsigned long long tmo = args.timeout_ns;
    int* const err = args.err;
    const int n_mma = args.n_mma;
    const int units = args.n_tiles * args.splits;

    const uint32_t bar0 = base + SK_OFF_BAR;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (SK_STAGES + s); };
    auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * SK_STAGES + b); };
    auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * SK_STAGES + 2 + b); };
    const uint32_t drain_bar = bar0 + 8u * (SK_NUM_BARS - 1);
    volatile uint32_t* tmem_holder = reinterpret_cast<volatile uint32_t*>(base_ptr + SK_OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + SK_OFF_MISC + 4);

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < SK_STAGES; ++s) {
            ptx::mbar_init(full_bar(s), 1);
            ptx::mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(tfull_bar(b), 1);
            ptx::mbar_init(tempty_bar(b), 4);
        }
        ptx::mbar_init(drain_bar, 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&args.w);
        ptx::prefetch_tmap(&args.x);
        ptx::prefetch_tmap(&args.out);
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32((const void*)tmem_holder), SK_TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    // work unit u: weight rows [128 * (u % n_tiles), +128), k-blocks of split u / n_tiles
    auto unit_range = [&](int u, int& n0, int& kb0, int& kb1) {
        const int tile = u % args.n_tiles;
        const int split = u / args.n_tiles;
        n0 = tile * BM;
        kb0 = split * args.kb_per_split;
        kb1 = min(args.k_blocks, kb0 + args.kb_per_split);
    };

    if (warp == 0) {
        if (lane == 0 && !(args.debug_flags & DEBUG_SKIP_PRODUCER)) {
            int stage = 0;
            uint32_t phase = 0;
            int last_parity[SK_STAGES];
            for (int s = 0; s < SK_STAGES; ++s) last_parity[s] = -1;
            const uint32_t tx = SK_A_BYTES + (uint32_t)n_mma * BK * 2;
            const bool w_mn = args.w_mn != 0;
            bool ok = true;
            for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
                int n0, kb0, kb1;
                unit_range(u, n0, kb0, kb1);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!wait_bounded(empty_bar(stage), phase ^ 1u, tmo, err, abort_flag, ERR_PRODUCER)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = full_bar(stage);
                    ptx::mbar_arrive_expect_tx(fb, tx);
                    last_parity[stage] = (int)phase;
                    const int k0 = kb * BKE;
                    const uint32_t sA = base + stage * SK_A_BYTES;
                    const uint32_t sB = base + SK_OFF_B + stage * SK_B_BYTES;
                    if (w_mn) {
                        ptx::tma_load_2d(sA, &args.w, fb, n0, k0);
                        ptx::tma_load_2d(sA + 8192, &args.w, fb, n0 + 64, k0);
                    } else {
                        ptx::tma_load_2d(sA, &args.w, fb, k0, n0);
                    }
                    ptx::tma_load_2d(sB, &args.x, fb, k0, 0);
                    if (++stage == SK_STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok)
                for (int s = 0; s < SK_STAGES; ++s)
                    if (last_parity[s] >= 0) drain_wait(full_bar(s), (uint32_t)last_parity[s], tmo);
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            const bool w_mn = args.w_mn != 0;
            const uint32_t fmt = OP == OP_E4M3 ? 0u : 1u;   // E4M3 or bf16
            const uint32_t idesc = (1u << 4) | (fmt << 7) | (fmt << 10) | ((w_mn ? 1u : 0u) << 15) |
                                   ((uint32_t)(n_mma >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            int local = 0;
            for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++local) {
                int n0, kb0, kb1;
                unit_range(u, n0, kb0, kb1);
                const int ab = local & 1;
                const uint32_t use = (uint32_t)(local >> 1);
                if (!wait_bounded(tempty_bar(ab), (use & 1u) ^ 1u, tmo, err, abort_flag, ERR_MMA)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(ab * SK_MAX_M);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!wait_bounded(full_bar(stage), phase, tmo, err, abort_flag, ERR_MMA)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t sA = base + stage * SK_A_BYTES;
                    const uint32_t sB = base + SK_OFF_B + stage * SK_B_BYTES;
#pragma unroll
                    for (int k = 0; k < BK / UMMA_K; ++k) {
                        const uint64_t ad = w_mn ? umma_desc_sw128(sA + k * 2048, 8192, 1024)
                                                 : umma_desc_sw128(sA + k * 32, 16, 1024);
                        const uint64_t bd = umma_desc_sw128(sB + k * 32, 16, 1024);
                        if (OP == OP_E4M3) ptx::mma_e4m3(d_tmem, ad, bd, idesc, (kb > kb0 || k > 0) ? 1u : 0u);
                        else ptx::mma_bf16(d_tmem, ad, bd, idesc, (kb > kb0 || k > 0) ? 1u : 0u);
                    }
                    ptx::mma_commit(empty_bar(stage));
                    if (++stage == SK_STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                ptx::mma_commit(tfull_bar(ab));
            }
            if (!ok) {
                ptx::mma_commit(drain_bar);
                drain_wait(drain_bar, 0, tmo);
            }
        }
        __syncwarp();
    } else if (warp >= EPI_WARP0) {
        const int wq = warp & 3;
        const uint32_t out_tile = base + SK_OFF_OUT + wq * SK_OUT_WARP;
        int local = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++local) {
            int n0, kb0, kb1;
            unit_range(u, n0, kb0, kb1);
            const int split = u / args.n_tiles;
            const int ab = local & 1;
            const uint32_t use = (uint32_t)(local >> 1);
            const bool got = __all_sync(0xffffffffu,
                                        wait_bounded(tfull_bar(ab), use & 1u, tmo, err, abort_flag, ERR_EPILOGUE));
            if (!got) {
                ok = false;
                break;
            }
            ptx::tc_fence_after();
            const uint32_t t_row = tmem_base + ((uint32_t)(32 * wq) << 16) + (uint32_t)(ab * SK_MAX_M);
            const int chunks = n_mma / 16;
            // the previous unit's stores must have read the staging tile
            if (lane == 0) ptx::bulk_wait_group_read<0>();
            __syncwarp();
            for (int c = 0; c < chunks; ++c) {
                uint32_t v[16];
                ptx::tmem_ld_32x32b_x16(t_row + c * 16, v);
                ptx::tmem_ld_wait();
                const uint32_t tile = out_tile + c * 2048;   // 32 rows x 16 fp32
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    ptx::sts128(tile + sw64_offset(lane, q), make_uint4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]));
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(tempty_bar(ab));
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0 && n0 + 32 * wq < args.N) {
                for (int c = 0; c < chunks; ++c)
                    ptx::tma_store_3d(&args.out, out_tile + c * 2048, 16 * c, n0 + 32 * wq, split);
            }
            if (lane == 0) ptx::bulk_commit_group();
        }
        if (lane == 0) ptx::bulk_wait_group<0>();
        ptx::tc_fence_before();
        __syncwarp();
    }
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, SK_TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------
// element-wise finishing kernels (fp32 [N, ld] transposed sums -> bf16 outputs)
// ---------------------------------------------------------------------------

// The fp32 partial planes of the split-K products: element (row n, token m) of the
// sum is the planes' values added in plane order (a fixed order: the same bits on
// every run).
struct Planes {
    const float* p;
    int ld;                // tokens per row (M rounded up to 16)
    int count;             // splits
    long long stride;      // elements per plane (rows * ld)
    __device__ __forceinline__ float at(long long row, int m) const {
        const float* q = p + row * ld + m;
        float s = q[0];
#pragma unroll 8
        for (int k = 1; k < count; ++k) s += q[k * stride];   // loads independent, adds in plane order
        return s;
    }
};

// out [M, N] bf16 = round(scale * acc^T (+ res)), res [M, N] bf16 optional (the
// residual block); scale is 1 except for FP8 sums
__global__ void skinny_cast_kernel(Planes acc, const __nv_bfloat16* __restrict__ res,
                                   __nv_bfloat16* __restrict__ out, int M, int N, float scale = 1.0f) {
    const long long total = (long long)M * N;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total; i += (long long)gridDim.x * blockDim.x) {
        const int m = (int)(i / N), n = (int)(i % N);
        const float r = res ? __bfloat162float(res[i]) : 0.0f;
        out[i] = __float2bfloat16_rn(scale * acc.at(n, m) + r);
    }
}

// FP8 SwiGLU forward from the unscaled fp32 sums preact^T [2H, ld]: preact [M, 2H]
// (optional, bf16 of scale_acc * sum) and h8 [M, H] = E4M3(h * inv_s_h), h from the
// bf16 preact as in the bf16 kernels; codes round to nearest even and saturate.
__global__ void skinny_swiglu_fwd_fp8_kernel(Planes acc, float scale_acc, float inv_s_h,
                                             __nv_bfloat16* __restrict__ preact, uint8_t* __restrict__ h8, int M,
                                             int H) {
    const long long total = (long long)M * H;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total; i += (long long)gridDim.x * blockDim.x) {
        const int m = (int)(i / H), j = (int)(i % H);
        const __nv_bfloat16 lb = __float2bfloat16_rn(scale_acc * acc.at(j, m));
        const __nv_bfloat16 gb = __float2bfloat16_rn(scale_acc * acc.at(H + j, m));
        if (preact) {
            preact[(long long)m * 2 * H + j] = lb;
            preact[(long long)m * 2 * H + H + j] = gb;
        }
        const float g = __bfloat162float(gb);
        const float hv = __bfloat162float(lb) * round_bf16(g * sigmoid_mufu(g));
        h8[i] = (uint8_t)(ptx::cvt_e4m3x2(hv * inv_s_h, 0.0f) & 0xFFu);
    }
}

// SwiGLU forward from the fp32 preact^T [2H, ld]: preact [M, 2H] and h [M, H],
// h = bf16(left * bf16(silu(gate))) with left, gate the bf16-rounded preact.
__global__ void skinny_swiglu_fwd_kernel(Planes acc, __nv_bfloat16* __restrict__ preact,
                                         __nv_bfloat16* __restrict__ h, int M, int H) {
    const long long total = (long long)M * H;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total; i += (long long)gridDim.x * blockDim.x) {
        const int m = (int)(i / H), j = (int)(i % H);
        const __nv_bfloat16 lb = __float2bfloat16_rn(acc.at(j, m));
        const __nv_bfloat16 gb = __float2bfloat16_rn(acc.at(H + j, m));
        preact[(long long)m * 2 * H + j] = lb;
        preact[(long long)m * 2 * H + H + j] = gb;
        const float g = __bfloat162float(gb);
        h[i] = __float2bfloat16_rn(__bfloat162float(lb) * round_bf16(g * sigmoid_mufu(g)));
    }
}

// SwiGLU backward from the fp32 grad_h^T [H, ld] and the saved preact:
// grad_preact [M, 2H] = [grad_h * silu(gate) | grad_h * left * silu'(gate)], h [M, H].
__global__ void skinny_swiglu_bwd_kernel(Planes acc, const __nv_bfloat16* __restrict__ preact,
                                         __nv_bfloat16* __restrict__ grad_preact, __nv_bfloat16* __restrict__ h, int M,
                                         int H) {
    const long long total = (long long)M * H;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total; i += (long long)gridDim.x * blockDim.x) {
        const int m = (int)(i / H), j = (int)(i % H);
        const float gh = acc.at(j, m);
        const float l = __bfloat162float(preact[(long long)m * 2 * H + j]);
        const float g = __bfloat162float(preact[(long long)m * 2 * H + H + j]);
        const float sig = sigmoid_mufu(g);
        const float silu = g * sig;
        const float silu_p = sig + silu * (1.0f - sig);
        grad_preact[(long long)m * 2 * H + j] = __float2bfloat16_rn(gh * silu);
        grad_preact[(long long)m * 2 * H + H + j] = __float2bfloat16_rn(gh * l * silu_p);
        h[i] = __float2bfloat16_rn(l * round_bf16(silu));
    }
}

}  // namespace swiglu
