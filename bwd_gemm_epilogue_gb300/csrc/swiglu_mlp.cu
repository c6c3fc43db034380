// swiglu_mlp.cu -- host side of the C ABI declared in include/swiglu_mlp.h:
// argument validation, TMA tensor-map encoding, persistent-grid sizing and the
// launches of the tcgen05 GEMM kernel variants (gemm_kernel.cuh).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <functional>
#include <queue>
#include <utility>
#include <vector>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "gemm_kernel.cuh"
#include "skinny_kernel.cuh"
#include "swiglu_mlp.h"
#include "swiglu_moe.h"

namespace swiglu {
namespace {

constexpr int kMaxDevices = 64;

__device__ int g_err_word;   // device error word: ERR_* bits of roles that gave up a wait

std::atomic<unsigned long long> g_timeout_ns{4000000000ull};
std::atomic<int> g_debug_flags{0};
std::atomic<int> g_raster_band{0};   // 0: the default band of 8 tiles

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct DeviceState {
    bool ready = false;
    int num_sms = 0;
    int* err_word = nullptr;
};

struct Trace {
    cudaEvent_t* events = nullptr;
    int* kinds = nullptr;
    int capacity = 0;
    int count = 0;
};
thread_local Trace g_trace;

// Last failure on this thread, for swiglu_mlp_last_error_detail.
thread_local char g_detail[256];

swiglu_status fail(swiglu_status st, const char* what, cudaError_t err = cudaSuccess) {
    if (err != cudaSuccess)
        std::snprintf(g_detail, sizeof g_detail, "%s: %s (%s)", what, cudaGetErrorName(err), cudaGetErrorString(err));
    else
        std::snprintf(g_detail, sizeof g_detail, "%s", what);
    return st;
}

std::mutex g_mutex;
EncodeTiledFn g_encode = nullptr;
DeviceState g_dev[kMaxDevices];

swiglu_status get_device_state(DeviceState** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) return fail(SWIGLU_ERR_CUDA, "cudaGetDevice", e);
    // A thread that has not used CUDA yet (an autograd worker, a fresh std::thread) has
    // no current context, and the tensor-map encoder needs one.  Binding the current
    // device's primary context is a no-op when it is already current.
    e = cudaSetDevice(dev);
    if (e != cudaSuccess) return fail(SWIGLU_ERR_CUDA, "cudaSetDevice", e);
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr)
            return fail(SWIGLU_ERR_CUDA, "cudaGetDriverEntryPointByVersion(cuTensorMapEncodeTiled)", e);
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    DeviceState& st = g_dev[dev];
    if (!st.ready) {
        e = cudaDeviceGetAttribute(&st.num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return fail(SWIGLU_ERR_CUDA, "cudaDeviceGetAttribute", e);
        e = cudaGetSymbolAddress(reinterpret_cast<void**>(&st.err_word), g_err_word);
        if (e != cudaSuccess) return fail(SWIGLU_ERR_CUDA, "cudaGetSymbolAddress(error word)", e);
        st.ready = true;
    }
    *out = &st;
    return SWIGLU_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// 2-D bf16 tensor map: `inner` contiguous elements per row, `outer` rows, row
// pitch `row_bytes`.
bool encode_2d(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t outer, uint64_t row_bytes,
               uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz,
               CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    return g_encode(m, dtype, 2, const_cast<void*>(ptr), dims, strides, box,
                    estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_3d(CUtensorMap* m, const void* ptr, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1_bytes,
               uint64_t s2_bytes, uint32_t b0, uint32_t b1, uint32_t b2, CUtensorMapSwizzle swz,
               CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {s1_bytes, s2_bytes};
    cuuint32_t box[3] = {b0, b1, b2};
    cuuint32_t estr[3] = {1, 1, 1};
    return g_encode(m, dtype, 3, const_cast<void*>(ptr), dims, strides, box,
                    estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Operand maps for the mainloop.  K-major: box 64 (k) x rows.  MN-major: box 64 (mn) x
// 64 (k), one copy per 64 rows -- or, when MN is a multiple of 64 and `three_d` is given,
// the 3-D view (64 mn, k, mn / 64) with box 64 x 64 x rows / 64, whose copy lands the
// same rows / 64 blocks of 8 KB in shared memory with a single instruction (*three_d is
// set then).  Fewer copies per k-block relieve the producer thread.
bool encode_operand(CUtensorMap* m, const void* ptr, int64_t mn, int64_t k, bool mn_major, uint32_t rows,
                    bool* three_d = nullptr) {
    if (three_d) *three_d = false;
    if (mn_major) {
        if (three_d && mn % 64 == 0 && rows >= 64 && rows % 64 == 0 &&
            encode_3d(m, ptr, 64, (uint64_t)k, (uint64_t)(mn / 64), (uint64_t)mn * 2, 128, 64, 64, rows / 64,
                      CU_TENSOR_MAP_SWIZZLE_128B)) {
            *three_d = true;
            return true;
        }
        return encode_2d(m, ptr, (uint64_t)mn, (uint64_t)k, (uint64_t)mn * 2, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B);
    }
    return encode_2d(m, ptr, (uint64_t)k, (uint64_t)mn, (uint64_t)k * 2, 64, rows, CU_TENSOR_MAP_SWIZZLE_128B);
}

// Epilogue tiles are `box_cols` bf16 wide: 32 columns (64-byte rows, 64-byte swizzle) or
// the fused backward's PRE_COLS = 64 (128-byte rows, 128-byte swizzle).
CUtensorMapSwizzle epi_swizzle(uint32_t box_cols) {
    return box_cols == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
}

// [M, 2H] tensor seen as (j, half, m): element (j, half, m) = base[m*2H + half*H + j].
bool encode_paired(CUtensorMap* m, const void* ptr, int64_t M, int64_t H, uint32_t box_rows,
                   uint32_t box_cols = CHUNK) {
    return encode_3d(m, ptr, (uint64_t)H, 2, (uint64_t)M, (uint64_t)H * 2, (uint64_t)H * 4, box_cols, 1, box_rows,
                     epi_swizzle(box_cols));
}

bool encode_out_2d(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, uint32_t box_cols = CHUNK) {
    return encode_2d(m, ptr, (uint64_t)cols, (uint64_t)rows, (uint64_t)cols * 2, box_cols, 32,
                     epi_swizzle(box_cols));
}

// Host-only test hook bit: run every GEMM with single-CTA tiles.
constexpr int DEBUG_FORCE_SINGLE_CTA = 2;

// CTA-pair tiles (256 rows) pay off once the GEMM has more than one 128-row tile.
int pick_cg(int64_t M) {
    if (g_debug_flags.load() & DEBUG_FORCE_SINGLE_CTA) return 1;
    return M > BM ? 2 : 1;
}

// Host-only test hook bit: the backward's dW2, dx and dW1 run as three launches.
constexpr int DEBUG_UNGROUPED = 4;

// Host-only test hook bits: plain GEMMs of CTA pairs always with 256 x 256 tiles, or
// with 256 x 512 tiles wherever N > 256 (instead of the choice below).
constexpr int DEBUG_NARROW_TILES = 32;
constexpr int DEBUG_WIDE_TILES = 64;
// Host-only test hook bit: no split tiles (see plan_split).
constexpr int DEBUG_NO_SPLIT = 128;

// slots: 2 for a problem of 256 x 512 tiles (EPI_STORE_W launches), else 1.
Problem make_problem(int64_t M, int64_t N, int64_t K, int64_t tiles_n, bool a_mn, bool b_mn, int cg, int slots = 1) {
    Problem p;
    p.M = (int)M;
    p.N = (int)N;
    p.K = (int)K;
    p.tiles_m = (int)((M + BM * cg - 1) / (BM * cg));
    p.tiles_n = (int)tiles_n;
    // raster band: 8 column tiles of 256 (2048 columns); 256 x 512 tiles take half as many
    int band = g_raster_band.load() > 0 ? g_raster_band.load() : 8;
    if (slots == 2) band = band > 1 ? band / 2 : 1;
    p.band = p.tiles_n < band ? p.tiles_n : band;
    p.k_blocks = (int)((K + BK - 1) / BK);
    p.a_mn = a_mn ? 1 : 0;
    p.b_mn = b_mn ? 1 : 0;
    p.a3d = 0;
    p.b3d = 0;
    p.res = 0;
    p.tile_begin = 0;
    p.no_o0 = 0;
    p.slots = slots;
    return p;
}

// A 256 x 512 tile's mainloop runs this much faster per FLOP than a 256 x 256 tile's (its
// k-blocks carry a quarter fewer operand bytes per FLOP), and the MMA issuer then waits
// about this many k-block times for the epilogue to read the previous tile's slots.
constexpr double kWideGain = 1.05;
constexpr double kWideDrain = 9.0;

// Time of one tile of problem p in 256 x 256 x 64 k-block times (the ragged last column
// tile of a 256 x 512 problem counted as a whole one).
double tile_cost(const Problem& p) {
    return p.slots == 2 ? 2.0 * p.k_blocks / kWideGain + kWideDrain : (double)p.k_blocks;
}

// Longest-processing-time assignment of the launch's tiles to `units` clusters:
// tiles in order of decreasing work (stable within a problem), each to the
// least-loaded cluster.  Returns false if the lists do not fit the parameter block.
bool build_schedule(ScheduledArgs& a, int units) {
    if (units > MAX_CLUSTERS || a.num_tiles > MAX_SCHED || a.num_tiles > 65535) return false;
    int order[MAX_PROBLEMS];
    for (int q = 0; q < a.num_problems; ++q) order[q] = q;
    std::stable_sort(order, order + a.num_problems,
                     [&](int x, int y) { return tile_cost(a.prob[x]) > tile_cost(a.prob[y]); });
    std::vector<std::vector<uint16_t>> lists(units);
    using Slot = std::pair<double, int>;   // (load, cluster)
    std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> heap;
    for (int u = 0; u < units; ++u) heap.push({0, u});
    for (int oi = 0; oi < a.num_problems; ++oi) {
        const Problem& p = a.prob[order[oi]];
        const int n = p.tiles_m * p.tiles_n;
        for (int t = 0; t < n; ++t) {
            Slot s = heap.top();
            heap.pop();
            lists[s.second].push_back((uint16_t)(p.tile_begin + t));
            heap.push({s.first + tile_cost(p), s.second});
        }
    }
    int off = 0;
    for (int u = 0; u < units; ++u) {
        a.sched_off[u] = (uint16_t)off;
        for (uint16_t t : lists[u]) a.sched[off++] = t;
    }
    a.sched_off[units] = (uint16_t)off;
    return true;
}

// Persistent CTAs (CG == 1) or CTA pairs (CG == 2) of this kernel that fit on the
// device at once; 0 on failure.
template <int EPI, int CG, int SCHED, int OP = OP_BF16>
int cluster_slots(DeviceState* st) {
    if (CG == 1) return st->num_sms;
    static int max_clusters[kMaxDevices];
    int dev = 0;
    cudaGetDevice(&dev);
    if (max_clusters[dev] <= 0) {
        auto kern = gemm_kernel<EPI, CG, SCHED, OP>;
        constexpr int smem = Cfg<EPI, CG>::SMEM_BYTES;
        // the occupancy query sees the kernel's dynamic shared memory limit
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return 0;
        cudaLaunchConfig_t cfg;
        std::memset(&cfg, 0, sizeof cfg);
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cfg.blockDim = dim3(Cfg<EPI, CG>::THREADS);
        cfg.dynamicSmemBytes = smem;
        cfg.gridDim = dim3(2 * (st->num_sms / 2));
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) return 0;
        max_clusters[dev] = n;
    }
    return max_clusters[dev];
}

// Launch `units` persistent clusters of the kernel over args (fields all filled in),
// bracketed by the launch trace's events when one is open.
template <int EPI, int CG, int SCHED, int OP = OP_BF16>
swiglu_status launch_grid(DeviceState* st, int kind, const ArgsOf<EPI, CG, SCHED>& args, int units,
                          cudaStream_t stream) {
    (void)st;
    auto kern = gemm_kernel<EPI, CG, SCHED, OP>;
    constexpr int smem = Cfg<EPI, CG>::SMEM_BYTES;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return fail(SWIGLU_ERR_LAUNCH, "cudaFuncSetAttribute(max dynamic smem)", e);
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cudaLaunchAttribute attr[1];
    cfg.blockDim = dim3(Cfg<EPI, CG>::THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    if (CG == 2) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    cfg.gridDim = dim3(units * CG);
    Trace& tr = g_trace;
    const int slot = tr.events ? tr.count++ : -1;
    const bool traced = slot >= 0 && slot < tr.capacity;
    if (traced) {
        tr.kinds[slot] = kind;
        e = cudaEventRecord(tr.events[2 * slot], stream);
        if (e != cudaSuccess) return fail(SWIGLU_ERR_CUDA, "cudaEventRecord(trace)", e);
    }
    e = cudaLaunchKernelEx(&cfg, kern, args);
    if (e != cudaSuccess) return fail(SWIGLU_ERR_LAUNCH, "cudaLaunchKernelEx", e);
    if (traced) {
        e = cudaEventRecord(tr.events[2 * slot + 1], stream);
        if (e != cudaSuccess) return fail(SWIGLU_ERR_CUDA, "cudaEventRecord(trace)", e);
    }
    return SWIGLU_OK;
}

// Launch one persistent grid over args' problems (parameter-block sources).  args'
// tensor maps and problems are filled in by the caller; this sets the common
// fields, the host schedule and the grid.
template <int EPI, int CG, int SCHED, int OP = OP_BF16>
swiglu_status launch(DeviceState* st, int kind, ArgsOf<EPI, CG, SCHED>& args, cudaStream_t stream) {
    static_assert(!is_table(SCHED), "table launches go through launch_table");
    int tiles = 0;
    for (int q = 0; q < args.num_problems; ++q) {
        args.prob[q].tile_begin = tiles;
        tiles += args.prob[q].tiles_m * args.prob[q].tiles_n;
    }
    args.num_tiles = tiles;
    args.timeout_ns = g_timeout_ns.load();
    args.err = st->err_word;
    args.debug_flags = g_debug_flags.load();
    const int slots = cluster_slots<EPI, CG, SCHED, OP>(st);
    if (slots <= 0) return fail(SWIGLU_ERR_LAUNCH, "cudaOccupancyMaxActiveClusters");
    const int units = tiles < slots ? tiles : slots;
    if constexpr (SCHED == SRC_PARAMS) {
        if (!build_schedule(args, units)) return fail(SWIGLU_ERR_UNSUPPORTED_SHAPE, "tile schedule too large");
    }
    return launch_grid<EPI, CG, SCHED, OP>(st, kind, args, units, stream);
}

// ---------------------------------------------------------------- small-M (decode) path

// Host-only test hook bit: keep the 128/256-row tile path even for M <= 64.
constexpr int DEBUG_NO_SKINNY = 8;

bool use_skinny(int64_t M) { return M >= 1 && M <= SK_MAX_M && !(g_debug_flags.load() & DEBUG_NO_SKINNY); }
int64_t skinny_ld(int64_t M) { return (M + 15) / 16 * 16; }

template <class F>
swiglu_status launch_traced(int kind, cudaStream_t stream, F&& do_launch) {
    Trace& tr = g_trace;
    const int slot = tr.events ? tr.count++ : -1;
    const bool traced = slot >= 0 && slot < tr.capacity;
    cudaError_t e;
    if (traced) {
        tr.kinds[slot] = kind;
        e = cudaEventRecord(tr.events[2 * slot], stream);
        if (e != cudaSuccess) return fail(SWIGLU_ERR_CUDA, "cudaEventRecord(trace)", e);
    }
    e = do_launch();
    if (e != cudaSuccess) return fail(SWIGLU_ERR_LAUNCH, "kernel launch", e);
    if (traced) {
        e = cudaEventRecord(tr.events[2 * slot + 1], stream);
        if (e != cudaSuccess) return fail(SWIGLU_ERR_CUDA, "cudaEventRecord(trace)", e);
    }
    return SWIGLU_OK;
}

// Split-K plan of one small-M product with N weight rows and reduction length K: the
// fewest splits whose makespan ceil(tiles * s / SMs) / s (in whole-K tiles) is within 2 %
// of the best over s = 1..32 with >= 2 k-blocks per split.  Planned for the GB300's 152
// SMs, so that the workspace queries (which see no device) and the launches agree.
constexpr int kPlanSms = 152;
struct SkinnyPlan {
    int n_tiles, k_blocks, kb_per_split, splits;
};
SkinnyPlan skinny_plan(int64_t N, int64_t K, bool fp8) {
    SkinnyPlan p;
    const int bke = fp8 ? 2 * BK : BK;
    p.n_tiles = (int)((N + BM - 1) / BM);
    p.k_blocks = (int)((K + bke - 1) / bke);
    auto span_of = [&](int sp) {
        const long long units = (long long)p.n_tiles * sp;
        return (double)((units + kPlanSms - 1) / kPlanSms) / sp;
    };
    double best = span_of(1);
    for (int sp = 2; sp <= 32 && sp * 2 <= p.k_blocks; ++sp) best = span_of(sp) < best ? span_of(sp) : best;
    int splits = 1;
    while (span_of(splits) > best * 1.02) ++splits;
    p.kb_per_split = (p.k_blocks + splits - 1) / splits;
    p.splits = (p.k_blocks + p.kb_per_split - 1) / p.kb_per_split;   // every split non-empty
    return p;
}

// Bytes of the fp32 partial planes [splits][N][M16] of one small-M product.
size_t skinny_acc_bytes(int64_t N, int64_t K, int64_t M, bool fp8) {
    return (size_t)skinny_plan(N, K, fp8).splits * (size_t)N * (size_t)skinny_ld(M) * 4;
}

// Partial planes of acc^T [N, M16] = W * X^T with W [N, K] (w_mn = 0) or [K, N] (w_mn = 1)
// and X [M, K]: work unit (tile, split) stores its 128 x M16 partial into plane `split`;
// *planes describes them for the element-wise kernels, which add them in plane order.
swiglu_status run_skinny(DeviceState* st, int kind, const void* W, bool w_mn, const void* X, float* acc, int64_t N,
                         int64_t K, int64_t M, cudaStream_t s, bool fp8, Planes* planes) {
    const int64_t ld = skinny_ld(M);
    static thread_local SkinnyArgs a;
    std::memset(&a, 0, sizeof a);
    if (fp8) {
        // E4M3 operands, K-major: 128 k values (bytes) per box row
        constexpr CUtensorMapDataType U8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
        if (w_mn || !encode_2d(&a.w, W, (uint64_t)K, (uint64_t)N, (uint64_t)K, 2 * BK, BM, CU_TENSOR_MAP_SWIZZLE_128B, U8))
            return fail(SWIGLU_ERR_LAUNCH, "tensor map encode (skinny fp8 w)");
        if (!encode_2d(&a.x, X, (uint64_t)K, (uint64_t)M, (uint64_t)K, 2 * BK, (uint32_t)ld, CU_TENSOR_MAP_SWIZZLE_128B, U8))
            return fail(SWIGLU_ERR_LAUNCH, "tensor map encode (skinny fp8 x)");
    } else {
        if (!encode_operand(&a.w, W, N, K, w_mn, BM)) return fail(SWIGLU_ERR_LAUNCH, "tensor map encode (skinny w)");
        if (!encode_operand(&a.x, X, M, K, false, (uint32_t)ld))
            return fail(SWIGLU_ERR_LAUNCH, "tensor map encode (skinny x)");
    }
    const SkinnyPlan plan = skinny_plan(N, K, fp8);
    {
        cuuint64_t dims[3] = {(cuuint64_t)ld, (cuuint64_t)N, (cuuint64_t)plan.splits};
        cuuint64_t strides[2] = {(cuuint64_t)ld * 4, (cuuint64_t)N * ld * 4};
        cuuint32_t box[3] = {16, 32, 1};
        cuuint32_t estr[3] = {1, 1, 1};
        if (g_encode(&a.out, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, acc, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return fail(SWIGLU_ERR_LAUNCH, "tensor map encode (skinny partial planes)");
    }
    a.N = (int)N;
    a.K = (int)K;
    a.n_mma = (int)ld;
    a.w_mn = w_mn ? 1 : 0;
    a.n_tiles = plan.n_tiles;
    a.k_blocks = plan.k_blocks;
    a.kb_per_split = plan.kb_per_split;
    a.splits = plan.splits;
    a.timeout_ns = g_timeout_ns.load();
    a.err = st->err_word;
    a.debug_flags = g_debug_flags.load();
    *planes = Planes{acc, (int)ld, plan.splits, (long long)N * ld};
    auto kern = fp8 ? skinny_gemm_kernel<OP_E4M3> : skinny_gemm_kernel<OP_BF16>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SK_SMEM_BYTES);
    if (e != cudaSuccess) return fail(SWIGLU_ERR_LAUNCH, "cudaFuncSetAttribute(skinny smem)", e);
    const int units = plan.n_tiles * plan.splits;
    const int grid = units < st->num_sms ? units : st->num_sms;
    return launch_traced(kind, s, [&]() {
        kern<<<grid, NUM_THREADS, SK_SMEM_BYTES, s>>>(a);
        return cudaGetLastError();
    });
}

int elementwise_grid(DeviceState* st, long long total) {
    long long g = (total + 255) / 256;
    const long long cap = (long long)st->num_sms * 8;
    return (int)(g < cap ? (g < 1 ? 1 : g) : cap);
}

struct SkinnyFwdWs { void* h; float* pt; float* yt; };
struct SkinnyBwdWs { void* h; void* gp; float* gt; float* dxt; };

size_t skinny_fwd_ws(int64_t M, int64_t D, int64_t H, int64_t Dout, SkinnyFwdWs* w, void* base);
size_t skinny_bwd_ws(int64_t M, int64_t D, int64_t H, int64_t Dout, SkinnyBwdWs* w, void* base);

bool dims_ok(int64_t v) { return v > 0 && v % 8 == 0 && v < (int64_t(1) << 31); }

size_t round256(size_t v) { return (v + 255) & ~size_t(255); }

// Workspace layouts of the small-M path: the regular buffers first (h; h and
// grad_preact), then the fp32 partial planes of the transposed products.
size_t skinny_fwd_ws(int64_t M, int64_t D, int64_t H, int64_t Dout, SkinnyFwdWs* w, void* base) {
    size_t off = 0;
    auto take = [&](size_t bytes) {
        uint8_t* p = base ? static_cast<uint8_t*>(base) + off : nullptr;
        off += round256(bytes);
        return p;
    };
    uint8_t* h = take((size_t)M * H * 2);
    uint8_t* pt = take(skinny_acc_bytes(2 * H, D, M, false));     // preact^T planes, K = D
    uint8_t* yt = take(skinny_acc_bytes(Dout, H, M, false));      // y^T planes, K = H
    if (w) *w = SkinnyFwdWs{h, reinterpret_cast<float*>(pt), reinterpret_cast<float*>(yt)};
    return off;
}

size_t skinny_bwd_ws(int64_t M, int64_t D, int64_t H, int64_t Dout, SkinnyBwdWs* w, void* base) {
    size_t off = 0;
    auto take = [&](size_t bytes) {
        uint8_t* p = base ? static_cast<uint8_t*>(base) + off : nullptr;
        off += round256(bytes);
        return p;
    };
    uint8_t* h = take((size_t)M * H * 2);
    uint8_t* gp = take((size_t)M * 2 * H * 2);
    uint8_t* gt = take(skinny_acc_bytes(H, Dout, M, false));      // grad_h^T planes, K = Dout
    uint8_t* dxt = take(skinny_acc_bytes(D, 2 * H, M, false));    // dx^T planes, K = 2H
    if (w) *w = SkinnyBwdWs{h, gp, reinterpret_cast<float*>(gt), reinterpret_cast<float*>(dxt)};
    return off;
}

// Forward for M <= 64 tokens.
swiglu_status run_fwd_skinny(DeviceState* st, const void* x, const void* W1, const void* W2, void* preact, void* y,
                             int64_t M, int64_t D, int64_t H, int64_t Dout, void* ws, cudaStream_t s,
                             bool residual) {
    SkinnyFwdWs w;
    skinny_fwd_ws(M, D, H, Dout, &w, ws);
    Planes pt, yt;
    swiglu_status rc = run_skinny(st, SWIGLU_KERNEL_FWD_PREACT, W1, false, x, w.pt, 2 * H, D, M, s, false, &pt);
    if (rc != SWIGLU_OK) return rc;
    const int g = elementwise_grid(st, (long long)M * H);
    rc = launch_traced(SWIGLU_KERNEL_ELEMENTWISE, s, [&]() {
        skinny_swiglu_fwd_kernel<<<g, 256, 0, s>>>(pt, static_cast<__nv_bfloat16*>(preact),
                                                    static_cast<__nv_bfloat16*>(w.h), (int)M, (int)H);
        return cudaGetLastError();
    });
    if (rc != SWIGLU_OK) return rc;
    rc = run_skinny(st, SWIGLU_KERNEL_FWD_DOWN, W2, false, w.h, w.yt, Dout, H, M, s, false, &yt);   // y^T
    if (rc != SWIGLU_OK) return rc;
    const int g2 = elementwise_grid(st, (long long)M * Dout);
    return launch_traced(SWIGLU_KERNEL_ELEMENTWISE, s, [&]() {
        skinny_cast_kernel<<<g2, 256, 0, s>>>(yt, residual ? static_cast<const __nv_bfloat16*>(x) : nullptr,
                                              static_cast<__nv_bfloat16*>(y), (int)M, (int)Dout);
        return cudaGetLastError();
    });
}

// ---------------------------------------------------------------- the block's kernels

// preact = x @ W1^T with the SwiGLU forward epilogue (writes preact and h).
swiglu_status run_fwd_preact(DeviceState* st, const void* x, const void* W1, void* preact, void* h,
                             int64_t M, int64_t D, int64_t H, cudaStream_t s) {
    const int cg = pick_cg(M);
    KernelArgs a;
    std::memset(&a, 0, sizeof a);
    if (!encode_operand(&a.a[0], x, M, D, false, BM)) return fail(SWIGLU_ERR_LAUNCH, "tensor map encode (a)");
    // W1 [2H, D] as (k, j, half): element (k, j, half) = W1[(half*H + j)*D + k]
    if (!encode_3d(&a.b[0], W1, (uint64_t)D, (uint64_t)H, 2, (uint64_t)D * 2, (uint64_t)H * D * 2, 64, BN / 2, 1,
                   CU_TENSOR_MAP_SWIZZLE_128B))
        return fail(SWIGLU_ERR_LAUNCH, "tensor map encode (W1 slabs)");
    if (!encode_paired(&a.o0[0], preact, M, H, 32)) return fail(SWIGLU_ERR_LAUNCH, "tensor map encode (o0)");
    if (!encode_out_2d(&a.o1, h, M, H)) return fail(SWIGLU_ERR_LAUNCH, "tensor map encode (o1)");
    a.num_problems = 1;
    a.prob[0] = make_problem(M, H, D, (H + BN / 2 - 1) / (BN / 2), false, false, cg);
    if (cg == 2) return launch<EPI_SWIGLU_FWD, 2, SRC_SINGLE>(st, SWIGLU_KERNEL_FWD_PREACT, a, s);
    return launch<EPI_SWIGLU_FWD, 1, SRC_SINGLE>(st, SWIGLU_KERNEL_FWD_PREACT, a, s);
}

// grad_h = dy @ W2 fused with the SwiGLU backward (writes grad_preact and h).
swiglu_status run_fused_bwd(DeviceState* st, const void* dy, const void* W2, const void* preact,
                            void* grad_preact, void* h, int64_t M, int64_t H, int64_t Dout, cudaStream_t s) {
    const int cg = pick_cg(M);
    KernelArgs a;
    std::memset(&a, 0, sizeof a);
    if (!encode_operand(&a.a[0], dy, M, Dout, false, BM)) return fail(SWIGLU_ERR_LAUNCH, "tensor map encode (a)");
    // B(n = j, k = o) = W2[o, j]: MN-major
    bool b3d = false;
    if (!encode_operand(&a.b[0], W2, H, Dout, true, BN / cg, &b3d)) return fail(SWIGLU_ERR_LAUNCH, "tensor map encode (b)");
    // each epilogue warp moves 32 rows x PRE_COLS columns (128-byte rows) of preact and outputs
    if (!encode_paired(&a.o0[0], grad_preact, M, H, 32, PRE_COLS)) return fail(SWIGLU_ERR_LAUNCH, "tensor map encode (o0)");
    if (!encode_out_2d(&a.o1, h, M, H, PRE_COLS)) return fail(SWIGLU_ERR_LAUNCH, "tensor map encode (o1)");
    if (!encode_paired(&a.i0, preact, M, H, 32, PRE_COLS)) return fail(SWIGLU_ERR_LAUNCH, "tensor map encode (i0)");
    a.num_problems = 1;
    a.prob[0] = make_problem(M, H, Dout, (H + BN - 1) / BN, false, true, cg);
    a.prob[0].b3d = b3d ? 1 : 0;
    if (cg == 2) return launch<EPI_SWIGLU_BWD, 2, SRC_SINGLE>(st, SWIGLU_KERNEL_BWD_GRAD_H, a, s);
    return launch<EPI_SWIGLU_BWD, 1, SRC_SINGLE>(st, SWIGLU_KERNEL_BWD_GRAD_H, a, s);
}

struct GemmSpec {
    const void* A;
    const void* B;
    void* C;
    int64_t M, N, K;
    bool a_mn, b_mn;
    const void* R = nullptr;   // optional residual [M, N] added to C
};

// Fill problem q of `a`: C [M,N] = A * B^T (+ R) with either operand K-major or MN-major.
// A residual goes through the launch's single residual map i0.
// 256 x 512 tiles against 256 x 256 tiles.  A wide tile's k-blocks carry a quarter fewer
// operand bytes per FLOP: the tensor pipe runs faster while fed (with twice the MMA work
// per operand byte it ran 12-15 % faster at 11136 x 3584 x 14336, 11136 x 3584 x 28672 and
// 8192^3) and a FLOP costs less energy, which counts double while the step runs at the
// power cap.  But a wide tile holds both TMEM accumulators, so the MMA issuer waits for the
// epilogue to read the previous tile's slots, and the tile count halves.  The rules below
// are fitted to steps measured with each choice (narrow / chosen / wide everywhere):
//   target block (11136 tokens)   6549 / 6211 / 6135 us
//   8 experts of 2048 rows          11774 / 11142 / 11017 us
//   4096-token block                1984 / 1990 / 2000 us (its grouped backward loses 1.5 %,
//                                   its down projection gains 4 %)
//   64 experts of ~384 rows         1311 / 1311 / 1289 us (grouped backward 681 -> 656 us,
//                                   down projection 130 -> 135 us)
// The backward's dW2 / dx / dW1 group, longest-first over the parameter block: wide if there
// are at least kWideMinClusterKBlocks k-block times of work per CTA pair, at least
// kWideMinKBlocks per 256 x 256 tile on average (the 4096-token block's group, mostly tiles of
// 64 k-blocks, is not), and the longest wide tile fits the even share.  The same group over a table of experts: wide tiles always (half the tiles means
// half the per-tile problem switches, which cost more there than the slot reads).
constexpr double kWideMinKBlocks = 100;
constexpr double kWideMinClusterKBlocks = 2000;
// Down projections and other single products: wide if their reduction is long (at least
// kWideMinKBlocksLong k-blocks per tile, so the exposed slot reads stay near 1 % of a tile)
// and the wide tiles still fill every CTA pair once.
constexpr double kWideMinKBlocksLong = 100;

struct WideStats {
    double work = 0, tiles = 0, longest = 0, wide_tiles = 0;
};
WideStats wide_stats(const GemmSpec* g, int n) {
    WideStats w;
    for (int q = 0; q < n; ++q) {
        const double kb = (double)((g[q].K + BK - 1) / BK);
        const double tm = (double)((g[q].M + 2 * BM - 1) / (2 * BM));
        w.work += kb * tm * (double)((g[q].N + BN - 1) / BN);
        w.tiles += tm * (double)((g[q].N + BN - 1) / BN);
        w.wide_tiles += tm * (double)((g[q].N + 2 * BN - 1) / (2 * BN));
        w.longest = kb > w.longest ? kb : w.longest;
    }
    return w;
}

enum WideRule { WIDE_GROUP, WIDE_TABLE_GROUP, WIDE_LONG_K };
bool wide_pays(DeviceState* st, const GemmSpec* g, int n, WideRule rule) {
    const int flags = g_debug_flags.load();
    if (flags & DEBUG_NARROW_TILES) return false;
    bool any = false;
    for (int q = 0; q < n; ++q) any = any || g[q].N > BN;
    if (!any) return false;
    if ((flags & DEBUG_WIDE_TILES) || rule == WIDE_TABLE_GROUP) return true;
    const int units = cluster_slots<EPI_STORE, 2, SRC_SINGLE>(st);
    if (units <= 0) return false;
    const WideStats w = wide_stats(g, n);
    if (rule == WIDE_LONG_K) return w.work >= kWideMinKBlocksLong * w.tiles && w.wide_tiles >= units;
    return w.work >= kWideMinClusterKBlocks * units && w.work >= kWideMinKBlocks * w.tiles &&
           2 * w.longest <= w.work / units;
}

// wide: 256 x 512 tiles (EPI_STORE_W launches).
bool add_problem(KernelArgs& a, int q, const GemmSpec& g, int cg, bool wide = false) {
    bool a3d = false, b3d = false;
    if (!encode_operand(&a.a[q], g.A, g.M, g.K, g.a_mn, BM, &a3d)) return false;
    if (!encode_operand(&a.b[q], g.B, g.N, g.K, g.b_mn, BN / cg, &b3d)) return false;
    if (!encode_out_2d(&a.o0[q], g.C, g.M, g.N)) return false;
    const int64_t tile_n = wide ? 2 * BN : BN;
    a.prob[q] = make_problem(g.M, g.N, g.K, (g.N + tile_n - 1) / tile_n, g.a_mn, g.b_mn, cg, wide ? 2 : 1);
    a.prob[q].a3d = a3d ? 1 : 0;
    a.prob[q].b3d = b3d ? 1 : 0;
    if (g.R) {
        if (!encode_2d(&a.i0, g.R, (uint64_t)g.N, (uint64_t)g.M, (uint64_t)g.N * 2, CHUNK, BM, CU_TENSOR_MAP_SWIZZLE_64B))
            return false;
        a.prob[q].res = 1;
    }
    return true;
}

// Rows of a single GEMM in 256 x 512 tiles (K-major A) to keep in those tiles when the rows
// after them run as 256 x 256 tiles in the same launch: with few wide tiles per CTA pair the
// last round of a launch of wide tiles can be nearly empty (the target block's down
// projection: 308 tiles = 4.05 rounds over 76 pairs), and narrow tiles fill it.  The rows
// (all of M, or a multiple of 256) whose longest-first schedule has the shortest makespan in
// tile_cost units; 0 when plain 256 x 256 tiles do best.  Cached per shape and thread.
int64_t wide_rows(DeviceState* st, int64_t M, int64_t N, int64_t K) {
    const int units = cluster_slots<EPI_STORE_W, 2, SRC_PARAMS>(st);
    const int64_t tm = (M + 2 * BM - 1) / (2 * BM), tn_n = (N + BN - 1) / BN, tn_w = (N + 2 * BN - 1) / (2 * BN);
    if (units <= 0 || units > MAX_CLUSTERS || tm * tn_w >= 8LL * units || tm * tn_n > MAX_SCHED) return M;
    struct Entry {
        int64_t M, N, K;
        int units;
        int64_t rows;
    };
    thread_local std::vector<Entry> cache;
    for (const Entry& e : cache)
        if (e.M == M && e.N == N && e.K == K && e.units == units) return e.rows;
    const double kb = (double)((K + BK - 1) / BK);
    const double cw = 2.0 * kb / kWideGain + kWideDrain, cn = kb;
    double best = 0;
    int64_t best_a = tm;
    for (int64_t a = tm; a >= 0 && a >= tm - 16; --a) {
        std::priority_queue<double, std::vector<double>, std::greater<double>> load;
        for (int u = 0; u < units; ++u) load.push(0.0);
        auto put = [&](double c, int64_t n) {
            for (int64_t i = 0; i < n; ++i) {
                const double l = load.top();
                load.pop();
                load.push(l + c);
            }
        };
        put(cw, a * tn_w);       // longest tiles first, as build_schedule does
        put(cn, (tm - a) * tn_n);
        double ms = 0;
        for (; !load.empty(); load.pop()) ms = std::max(ms, load.top());
        if (a == tm || ms < best * (1 - 1e-9)) {
            best = ms;
            best_a = a;
        }
    }
    const int64_t rows = best_a >= tm ? M : best_a * 2 * BM;
    if (cache.size() >= 64) cache.erase(cache.begin());
    cache.push_back(Entry{M, N, K, units, rows});
    return rows;
}

// ---------------------------------------------------------------- split tiles
// Pieces of split tiles are at least this many k-blocks long: a boundary that would cut a
// shorter piece moves to the tile's edge.
constexpr int kSplitMinPiece = 8;
constexpr size_t kSplitFlagBytes = (size_t)MAX_SPLIT * SPLIT_UNITS * 2 * sizeof(int);

// Workspace bytes the split tiles of one K-major GEMM in 256 x 512 tiles may use: the
// counter pairs, then the fp32 sums ([MAX_SPLIT][SPLIT_UNITS][32 x SPLIT_COLS]).  Nonzero
// where such a launch can have them: M >= 256, N a multiple of 512, a long reduction (the
// rule for 256 x 512 tiles) and at least kSplitMinTiles tiles.
constexpr int64_t kSplitMinTiles = 144;
size_t split_ws_bytes(int64_t M, int64_t N, int64_t K) {
    if (M < 2 * BM || N <= 0 || N % (2 * BN) != 0 || (double)((K + BK - 1) / BK) < kWideMinKBlocksLong) return 0;
    if ((M + 2 * BM - 1) / (2 * BM) * (N / (2 * BN)) < kSplitMinTiles) return 0;
    return round256(kSplitFlagBytes) + (size_t)MAX_SPLIT * SPLIT_UNITS * SPLIT_UNIT_FLOATS * sizeof(float);
}

// Host lists for one GEMM in 256 x 512 tiles (a.prob[0], every tile with both slots).
// Whole tiles go round robin for all rounds but the last; the k-blocks of the tiles left
// (between one and two rounds of them) are then divided evenly over the `units` CTA
// pairs, each pair taking a contiguous run of (tile, k-block).  A tile that a boundary cuts
// is a split tile: its prefix piece (k-blocks [0, r)) ends one pair's run and its suffix
// piece ([r, kb)) starts the next one's.  Longest-first lists of whole tiles leave the last
// round of a launch with few long tiles per pair partly idle (the target block's down
// projection: 308 tiles over 76 pairs = 4.05 rounds); split tiles fill it.  Every pair
// runs its prefix piece first and its suffix piece last: all pairs start the tail at
// k-block 0, and a pair's suffix piece starts at about the k-block the others reach at
// that time, so concurrent tiles keep reading the same k-slices of A and B (running one
// pair's suffix first instead put the pairs at staggered k-blocks: 36 % more DRAM reads).
// At least two rounds of tiles: a launch made of pieces alone (the 4096-token block's
// down projection: 128 tiles over 76 pairs) measured 3.6 % slower than whole tiles with a
// partly idle second round.  Returns the number of split tiles,
// or -1 where this plan does not apply (fewer than two rounds of tiles, a boundary that
// would leave a tile with three pieces, or lists that do not fit the parameter block).
int plan_split(ScheduledArgs& a, int units) {
    const Problem& p = a.prob[0];
    const int n = p.tiles_m * p.tiles_n, kb = p.k_blocks;
    if (a.num_problems != 1 || p.slots != 2 || p.N % (2 * BN) != 0) return -1;
    if (units < 2 || units > MAX_CLUSTERS || n < 2 * units || n + MAX_SPLIT > MAX_SCHED) return -1;
    if (kb < 4 * kSplitMinPiece || kb > 65535) return -1;
    const int t0 = (n / units - 1) * units;        // tiles of the whole rounds
    const int64_t S = (int64_t)(n - t0) * kb;      // k-blocks after them
    std::vector<int64_t> b(units + 1);
    for (int u = 0; u <= units; ++u) {
        int64_t v = (S * u + units / 2) / units;
        const int64_t r = v % kb;
        if (r > 0 && r < kSplitMinPiece) v -= r;
        else if (r > kb - kSplitMinPiece) v += kb - r;
        b[u] = v;
    }
    std::vector<int> id(n - t0, -1);
    int n_split = 0;
    for (int u = 1; u <= units; ++u) {
        if (b[u] <= b[u - 1]) return -1;           // every pair gets k-blocks
        if (b[u] % kb == 0) continue;
        const int t = (int)(b[u] / kb);
        if (id[t] >= 0) return -1;                 // a second boundary in one tile
        id[t] = n_split++;
    }
    if (n_split > MAX_SPLIT) return -1;
    std::vector<std::vector<uint16_t>> lists(units);
    for (int t = 0; t < t0; ++t) lists[t % units].push_back((uint16_t)t);
    for (int u = 0; u < units; ++u) {
        const int64_t lo = b[u], hi = b[u + 1];
        const int ta = (int)(lo / kb), oa = (int)(lo % kb);
        const int tb = (int)((hi - 1) / kb), ob = (int)(hi - (int64_t)tb * kb);
        const bool suffix = oa > 0, prefix = ob < kb;
        a.split[u][0] = SplitPiece{(uint16_t)oa, (uint16_t)kb, (uint16_t)(suffix ? id[ta] : 0), 0};
        a.split[u][1] = SplitPiece{0, (uint16_t)ob, (uint16_t)(prefix ? id[tb] : 0), 0};
        const uint16_t suf = (uint16_t)((t0 + ta) | SCHED_PIECE);
        const uint16_t pre = (uint16_t)((t0 + tb) | SCHED_PIECE | SCHED_PIECE_PREFIX);
        std::vector<uint16_t>& L = lists[u];
        if (prefix) L.push_back(pre);
        for (int t = suffix ? ta + 1 : ta; t < (prefix ? tb : tb + 1); ++t) L.push_back((uint16_t)(t0 + t));
        if (suffix) L.push_back(suf);
    }
    int off = 0;
    for (int u = 0; u < units; ++u) {
        a.sched_off[u] = (uint16_t)off;
        for (uint16_t t : lists[u]) a.sched[off++] = t;
    }
    a.sched_off[units] = (uint16_t)off;
    return n_split;
}

// One K-major GEMM in 256 x 512 tiles (EPI_STORE_W, or EPI_STORE_ADD_W with g's residual)
// with split tiles at the end of the launch (plan_split), the split tiles' counters and sums
// in split_ws (split_ws_bytes of them).  Returns SWIGLU_ERR_UNSUPPORTED_SHAPE, having
// enqueued nothing, where the plan does not apply.
template <int EPI>
swiglu_status launch_split(DeviceState* st, int kind, const GemmSpec& g, void* split_ws, cudaStream_t s) {
    static thread_local ScheduledArgs a;
    std::memset(static_cast<KernelArgs*>(&a), 0, sizeof(KernelArgs));
    if (!add_problem(a, 0, g, 2, true)) return fail(SWIGLU_ERR_LAUNCH, "tensor map encode (gemm)");
    a.num_problems = 1;
    a.prob[0].tile_begin = 0;
    a.num_tiles = a.prob[0].tiles_m * a.prob[0].tiles_n;
    const int slots = cluster_slots<EPI, 2, SRC_PARAMS>(st);
    if (slots <= 0) return fail(SWIGLU_ERR_LAUNCH, "cudaOccupancyMaxActiveClusters");
    const int units = a.num_tiles < slots ? a.num_tiles : slots;
    const int n_split = plan_split(a, units);
    if (n_split < 0) return SWIGLU_ERR_UNSUPPORTED_SHAPE;
    a.timeout_ns = g_timeout_ns.load();
    a.err = st->err_word;
    a.debug_flags = g_debug_flags.load();
    a.split_flags = static_cast<int*>(split_ws);
    a.split_sums = reinterpret_cast<float*>(static_cast<uint8_t*>(split_ws) + round256(kSplitFlagBytes));
    if (n_split > 0) {
        const cudaError_t e = cudaMemsetAsync(a.split_flags, 0, (size_t)n_split * SPLIT_UNITS * 2 * sizeof(int), s);
        if (e != cudaSuccess) return fail(SWIGLU_ERR_CUDA, "cudaMemsetAsync(split counters)", e);
    }
    return launch_grid<EPI, 2, SRC_PARAMS>(st, kind, a, units, s);
}

// One plain GEMM, optionally with a residual added in its epilogue.  split_ws: room for
// split tiles (split_ws_bytes(M, N, K) bytes), or null.
swiglu_status run_gemm(DeviceState* st, int kind, const void* A, const void* B, void* Cp, int64_t M, int64_t N,
                       int64_t K, bool a_mn, bool b_mn, cudaStream_t s, const void* R = nullptr,
                       void* split_ws = nullptr) {
    const int cg = pick_cg(M);
    KernelArgs a;
    std::memset(&a, 0, sizeof a);
    GemmSpec g{A, B, Cp, M, N, K, a_mn, b_mn};
    g.R = R;
    const bool wide_ok = cg == 2 && wide_pays(st, &g, 1, WIDE_LONG_K);
    if (wide_ok && split_ws && !a_mn && split_ws_bytes(M, N, K) > 0 &&
        !(g_debug_flags.load() & (DEBUG_NO_SPLIT | DEBUG_WIDE_TILES))) {
        const swiglu_status rc = R ? launch_split<EPI_STORE_ADD_W>(st, kind, g, split_ws, s)
                                   : launch_split<EPI_STORE_W>(st, kind, g, split_ws, s);
        if (rc != SWIGLU_ERR_UNSUPPORTED_SHAPE) return rc;
    }
    bool wide = !R && wide_ok;
    const int64_t rows = wide && !a_mn && !(g_debug_flags.load() & DEBUG_WIDE_TILES) ? wide_rows(st, M, N, K) : M;
    if (rows == 0) wide = false;
    if (wide && rows < M) {
        // the first `rows` rows in 256 x 512 tiles, the rest in 256 x 256 tiles, one launch
        static thread_local ScheduledArgs sa;
        std::memset(static_cast<KernelArgs*>(&sa), 0, sizeof(KernelArgs));
        const GemmSpec g1{static_cast<const uint8_t*>(A) + rows * K * 2, B, static_cast<uint8_t*>(Cp) + rows * N * 2,
                          M - rows, N, K, a_mn, b_mn};
        GemmSpec g0 = g;
        g0.M = rows;
        if (!add_problem(sa, 0, g0, 2, true) || !add_problem(sa, 1, g1, 2, false))
            return fail(SWIGLU_ERR_LAUNCH, "tensor map encode (gemm)");
        sa.num_problems = 2;
        return launch<EPI_STORE_W, 2, SRC_PARAMS>(st, kind, sa, s);
    }
    if (!add_problem(a, 0, g, cg, wide)) return fail(SWIGLU_ERR_LAUNCH, "tensor map encode (gemm)");
    a.num_problems = 1;
    if (R) {
        if (cg == 2) return launch<EPI_STORE_ADD, 2, SRC_SINGLE>(st, kind, a, s);
        return launch<EPI_STORE_ADD, 1, SRC_SINGLE>(st, kind, a, s);
    }
    if (wide) return launch<EPI_STORE_W, 2, SRC_SINGLE>(st, kind, a, s);
    if (cg == 2) return launch<EPI_STORE, 2, SRC_SINGLE>(st, kind, a, s);
    return launch<EPI_STORE, 1, SRC_SINGLE>(st, kind, a, s);
}

// Several independent plain GEMMs in one persistent launch, tiles balanced across
// the CTA pairs by the host schedule (CTA-pair tiles; all M > 128).  At most one of
// them may carry a residual.
swiglu_status run_gemm_group(DeviceState* st, int kind, const GemmSpec* g, int n, cudaStream_t s) {
    static thread_local ScheduledArgs a;   // ~26 KB: not on the stack
    std::memset(static_cast<KernelArgs*>(&a), 0, sizeof(KernelArgs));
    bool res = false;
    for (int q = 0; q < n; ++q) {
        if (g[q].R && res) return fail(SWIGLU_ERR_INVALID_ARG, "group: more than one residual");
        res = res || g[q].R != nullptr;
    }
    const bool wide = wide_pays(st, g, n, WIDE_GROUP);
    for (int q = 0; q < n; ++q)
        if (!add_problem(a, q, g[q], 2, wide)) return fail(SWIGLU_ERR_LAUNCH, "tensor map encode (group)");
    a.num_problems = n;
    if (res && wide) return launch<EPI_STORE_ADD_W, 2, SRC_PARAMS>(st, kind, a, s);
    if (res) return launch<EPI_STORE_ADD, 2, SRC_PARAMS>(st, kind, a, s);
    if (wide) return launch<EPI_STORE_W, 2, SRC_PARAMS>(st, kind, a, s);
    return launch<EPI_STORE, 2, SRC_PARAMS>(st, kind, a, s);
}

}  // namespace
}  // namespace swiglu

using namespace swiglu;

extern "C" {

size_t swiglu_mlp_fwd_workspace_size(int64_t M, int64_t D, int64_t H, int64_t Dout) {
    (void)D;
    if (M <= 0 || H <= 0) return 0;
    if (M <= SK_MAX_M && Dout > 0 && D > 0) return skinny_fwd_ws(M, D, H, Dout, nullptr, nullptr);
    return round256((size_t)M * (size_t)H * 2) + split_ws_bytes(M, Dout, H);
}

size_t swiglu_mlp_bwd_workspace_size(int64_t M, int64_t D, int64_t H, int64_t Dout) {
    (void)Dout;
    if (M <= 0 || H <= 0) return 0;
    if (M <= SK_MAX_M && D > 0 && Dout > 0) return skinny_bwd_ws(M, D, H, Dout, nullptr, nullptr);
    return round256((size_t)M * (size_t)H * 2) + round256((size_t)M * (size_t)H * 4);
}

static swiglu_status fwd_impl(const void* x, const void* W1, const void* W2, void* preact, void* y, int64_t M,
                              int64_t D, int64_t H, int64_t Dout, void* workspace, size_t workspace_bytes,
                              void* stream, bool residual) {
    if (M < 0 || D <= 0 || H <= 0 || Dout <= 0) return fail(SWIGLU_ERR_INVALID_ARG, "forward: a size is negative or zero");
    if (!dims_ok(D) || !dims_ok(H) || !dims_ok(Dout) || M >= (int64_t(1) << 31) || 2 * H >= (int64_t(1) << 31))
        return fail(SWIGLU_ERR_UNSUPPORTED_SHAPE, "forward: unsupported shape (widths must be positive multiples of 8 below 2^31)");
    if (M == 0) return SWIGLU_OK;
    if (!x || !W1 || !W2 || !preact || !y || !workspace) return fail(SWIGLU_ERR_INVALID_ARG, "forward: a required pointer is null");
    if (!aligned16(x) || !aligned16(W1) || !aligned16(W2) || !aligned16(preact) || !aligned16(y) ||
        !aligned16(workspace))
        return fail(SWIGLU_ERR_MISALIGNED, "forward: a pointer is not 16-byte aligned");
    if (workspace_bytes < swiglu_mlp_fwd_workspace_size(M, D, H, Dout)) return fail(SWIGLU_ERR_WORKSPACE_TOO_SMALL, "forward: workspace smaller than the size query returns");
    DeviceState* st;
    swiglu_status rc = get_device_state(&st);
    if (rc != SWIGLU_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (use_skinny(M)) return run_fwd_skinny(st, x, W1, W2, preact, y, M, D, H, Dout, workspace, s, residual);
    void* h = workspace;
    rc = run_fwd_preact(st, x, W1, preact, h, M, D, H, s);
    if (rc != SWIGLU_OK) return rc;
    // y = h @ W2^T (+ x for the residual block, added in the epilogue); split tiles' sums after h
    void* split = split_ws_bytes(M, Dout, H) ? static_cast<uint8_t*>(workspace) + round256((size_t)M * (size_t)H * 2)
                                             : nullptr;
    return run_gemm(st, SWIGLU_KERNEL_FWD_DOWN, h, W2, y, M, Dout, H, false, false, s, residual ? x : nullptr,
                    split);
}

swiglu_status swiglu_mlp_fwd(const void* x, const void* W1, const void* W2, void* preact, void* y, int64_t M,
                             int64_t D, int64_t H, int64_t Dout, void* workspace, size_t workspace_bytes,
                             void* stream) {
    return fwd_impl(x, W1, W2, preact, y, M, D, H, Dout, workspace, workspace_bytes, stream, false);
}

swiglu_status swiglu_mlp_fwd_residual(const void* x, const void* W1, const void* W2, void* preact, void* y,
                                      int64_t M, int64_t D, int64_t H, int64_t Dout, void* workspace,
                                      size_t workspace_bytes, void* stream) {
    if (D != Dout) return fail(SWIGLU_ERR_UNSUPPORTED_SHAPE, "residual block needs D == Dout");
    return fwd_impl(x, W1, W2, preact, y, M, D, H, Dout, workspace, workspace_bytes, stream, true);
}

// Records `event` (a cudaEvent_t, may be NULL) on `s`.
static swiglu_status record_event(void* event, cudaStream_t s) {
    if (!event) return SWIGLU_OK;
    cudaError_t e = cudaEventRecord(static_cast<cudaEvent_t>(event), s);
    return e == cudaSuccess ? SWIGLU_OK : fail(SWIGLU_ERR_CUDA, "cudaEventRecord", e);
}

// This thread's second stream on the current device, with an event to fork work onto it and
// one to join it back (per thread, so concurrent callers never share them).
static swiglu_status side_stream(cudaStream_t* side, cudaEvent_t* fork, cudaEvent_t* join) {
    struct Side {
        cudaStream_t s = nullptr;
        cudaEvent_t fork = nullptr, join = nullptr;
    };
    thread_local Side per_dev[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) return fail(SWIGLU_ERR_CUDA, "cudaGetDevice", e);
    Side& d = per_dev[dev];
    if (!d.s) {
        e = cudaStreamCreateWithFlags(&d.s, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&d.fork, cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&d.join, cudaEventDisableTiming);
        if (e != cudaSuccess) {
            d.s = nullptr;
            return fail(SWIGLU_ERR_CUDA, "a second stream of the calling thread", e);
        }
    }
    *side = d.s;
    *fork = d.fork;
    *join = d.join;
    return SWIGLU_OK;
}

// dx_event (tensor-parallel backward): when set, dx is computed by a launch of its own and
// the event is recorded after it, while the weight gradients run beside it on a second
// stream, so that a caller can reduce dx across ranks while dW1 and dW2 are computed.
static swiglu_status bwd_impl(const void* x, const void* W1, const void* W2, const void* preact, const void* dy,
                              void* dx, void* dW1, void* dW2, int64_t M, int64_t D, int64_t H, int64_t Dout,
                              void* workspace, size_t workspace_bytes, void* stream, bool residual,
                              void* dx_event = nullptr) {
    if (M < 0 || D <= 0 || H <= 0 || Dout <= 0) return fail(SWIGLU_ERR_INVALID_ARG, "backward: a size is negative or zero");
    if (!dims_ok(D) || !dims_ok(H) || !dims_ok(Dout) || M >= (int64_t(1) << 31) || 2 * H >= (int64_t(1) << 31))
        return fail(SWIGLU_ERR_UNSUPPORTED_SHAPE, "backward: unsupported shape (widths must be positive multiples of 8 below 2^31)");
    if (!W1 || !W2 || !dW1 || !dW2) return fail(SWIGLU_ERR_INVALID_ARG, "backward: a required pointer is null");
    if (!aligned16(W1) || !aligned16(W2) || !aligned16(dW1) || !aligned16(dW2)) return fail(SWIGLU_ERR_MISALIGNED, "backward: a pointer is not 16-byte aligned");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (M == 0) {
        cudaError_t e = cudaMemsetAsync(dW1, 0, (size_t)2 * H * D * 2, s);
        if (e == cudaSuccess) e = cudaMemsetAsync(dW2, 0, (size_t)Dout * H * 2, s);
        if (e != cudaSuccess) return fail(SWIGLU_ERR_CUDA, "cudaMemsetAsync", e);
        return record_event(dx_event, s);
    }
    if (!x || !preact || !dy || !dx || !workspace) return fail(SWIGLU_ERR_INVALID_ARG, "backward: a required pointer is null");
    if (!aligned16(x) || !aligned16(preact) || !aligned16(dy) || !aligned16(dx) || !aligned16(workspace))
        return fail(SWIGLU_ERR_MISALIGNED, "backward: a pointer is not 16-byte aligned");
    if (workspace_bytes < swiglu_mlp_bwd_workspace_size(M, D, H, Dout)) return fail(SWIGLU_ERR_WORKSPACE_TOO_SMALL, "backward: workspace smaller than the size query returns");
    DeviceState* st;
    swiglu_status rc = get_device_state(&st);
    if (rc != SWIGLU_OK) return rc;
    void* h = workspace;
    void* grad_preact = static_cast<uint8_t*>(workspace) + round256((size_t)M * (size_t)H * 2);
    if (use_skinny(M)) {
        // M <= 64 tokens: weight-streaming products transposed and split over K
        SkinnyBwdWs w;
        skinny_bwd_ws(M, D, H, Dout, &w, workspace);
        Planes gt, dxt;
        rc = run_skinny(st, SWIGLU_KERNEL_BWD_GRAD_H, W2, true, dy, w.gt, H, Dout, M, s, false, &gt);   // grad_h^T
        if (rc != SWIGLU_OK) return rc;
        const int ge = elementwise_grid(st, (long long)M * H);
        rc = launch_traced(SWIGLU_KERNEL_ELEMENTWISE, s, [&]() {
            skinny_swiglu_bwd_kernel<<<ge, 256, 0, s>>>(gt, static_cast<const __nv_bfloat16*>(preact),
                                                         static_cast<__nv_bfloat16*>(w.gp),
                                                         static_cast<__nv_bfloat16*>(w.h), (int)M, (int)H);
            return cudaGetLastError();
        });
        if (rc != SWIGLU_OK) return rc;
        rc = run_skinny(st, SWIGLU_KERNEL_BWD_DX, W1, true, w.gp, w.dxt, D, 2 * H, M, s, false, &dxt);   // dx^T
        if (rc != SWIGLU_OK) return rc;
        const int gc = elementwise_grid(st, (long long)M * D);
        rc = launch_traced(SWIGLU_KERNEL_ELEMENTWISE, s, [&]() {
            skinny_cast_kernel<<<gc, 256, 0, s>>>(dxt, residual ? static_cast<const __nv_bfloat16*>(dy) : nullptr,
                                                  static_cast<__nv_bfloat16*>(dx), (int)M, (int)D);
            return cudaGetLastError();
        });
        if (rc != SWIGLU_OK) return rc;
        rc = record_event(dx_event, s);
        if (rc != SWIGLU_OK) return rc;
        // the weight gradients (K = M) are output-bound: the regular kernels, as one launch when both use CTA pairs
        const GemmSpec wg[2] = {{dy, w.h, dW2, Dout, H, M, true, true}, {w.gp, x, dW1, 2 * H, D, M, true, true}};
        if (pick_cg(Dout) == 2 && pick_cg(2 * H) == 2 && !(g_debug_flags.load() & DEBUG_UNGROUPED))
            return run_gemm_group(st, SWIGLU_KERNEL_BWD_GEMMS, wg, 2, s);
        rc = run_gemm(st, SWIGLU_KERNEL_BWD_DW2, dy, w.h, dW2, Dout, H, M, true, true, s);
        if (rc != SWIGLU_OK) return rc;
        return run_gemm(st, SWIGLU_KERNEL_BWD_DW1, w.gp, x, dW1, 2 * H, D, M, true, true, s);
    }
    rc = run_fused_bwd(st, dy, W2, preact, grad_preact, h, M, H, Dout, s);
    if (rc != SWIGLU_OK) return rc;
    GemmSpec g[3] = {
        {dy, h, dW2, Dout, H, M, true, true},                 // dW2 = dy^T @ h
        {grad_preact, W1, dx, M, D, 2 * H, false, true},      // dx = grad_preact @ W1 (+ dy: residual block)
        {grad_preact, x, dW1, 2 * H, D, M, true, true},       // dW1 = grad_preact^T @ x (merged)
    };
    if (residual) g[1].R = dy;
    if (dx_event) {
        // dx in a launch of its own on `s`, the event after it; dW2 and dW1 (which do not read
        // dx; one launch when both use CTA pairs) on a second stream of this thread, so that
        // each launch's CTA pairs take the SMs the other one's last round leaves idle; `s`
        // waits for the second stream before the call returns
        cudaStream_t side;
        cudaEvent_t fork, join;
        rc = side_stream(&side, &fork, &join);
        if (rc != SWIGLU_OK) return rc;
        cudaError_t e = cudaEventRecord(fork, s);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(side, fork, 0);
        if (e != cudaSuccess) return fail(SWIGLU_ERR_CUDA, "backward: fork onto the second stream", e);
        rc = run_gemm(st, SWIGLU_KERNEL_BWD_DX, g[1].A, g[1].B, g[1].C, g[1].M, g[1].N, g[1].K, false, true, s, g[1].R);
        if (rc != SWIGLU_OK) return rc;
        rc = record_event(dx_event, s);
        if (rc != SWIGLU_OK) return rc;
        const GemmSpec wg[2] = {g[0], g[2]};
        int64_t wtiles = 0;
        for (const GemmSpec& q : wg) wtiles += ((q.M + 2 * BM - 1) / (2 * BM)) * ((q.N + BN - 1) / BN);
        if (!(g_debug_flags.load() & (DEBUG_UNGROUPED | DEBUG_FORCE_SINGLE_CTA)) && Dout > BM && 2 * H > BM &&
            wtiles <= MAX_SCHED) {
            rc = run_gemm_group(st, SWIGLU_KERNEL_BWD_GEMMS, wg, 2, side);
        } else {
            rc = run_gemm(st, SWIGLU_KERNEL_BWD_DW2, g[0].A, g[0].B, g[0].C, g[0].M, g[0].N, g[0].K, true, true, side);
            if (rc == SWIGLU_OK)
                rc = run_gemm(st, SWIGLU_KERNEL_BWD_DW1, g[2].A, g[2].B, g[2].C, g[2].M, g[2].N, g[2].K, true, true, side);
        }
        e = cudaEventRecord(join, side);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(s, join, 0);
        if (e != cudaSuccess) return fail(SWIGLU_ERR_CUDA, "backward: join the second stream", e);
        return rc;
    }
    int64_t pair_tiles = 0;   // tiles of the grouped launch (256-row CTA-pair tiles)
    for (const GemmSpec& q : g) pair_tiles += ((q.M + 2 * BM - 1) / (2 * BM)) * ((q.N + BN - 1) / BN);
    const bool grouped = !(g_debug_flags.load() & (DEBUG_UNGROUPED | DEBUG_FORCE_SINGLE_CTA)) && Dout > BM &&
                         M > BM && 2 * H > BM && pair_tiles <= MAX_SCHED;
    if (grouped) return run_gemm_group(st, SWIGLU_KERNEL_BWD_GEMMS, g, 3, s);
    rc = run_gemm(st, SWIGLU_KERNEL_BWD_DW2, g[0].A, g[0].B, g[0].C, g[0].M, g[0].N, g[0].K, true, true, s);
    if (rc != SWIGLU_OK) return rc;
    rc = run_gemm(st, SWIGLU_KERNEL_BWD_DX, g[1].A, g[1].B, g[1].C, g[1].M, g[1].N, g[1].K, false, true, s, g[1].R);
    if (rc != SWIGLU_OK) return rc;
    return run_gemm(st, SWIGLU_KERNEL_BWD_DW1, g[2].A, g[2].B, g[2].C, g[2].M, g[2].N, g[2].K, true, true, s);
}

swiglu_status swiglu_mlp_bwd(const void* x, const void* W1, const void* W2, const void* preact, const void* dy,
                             void* dx, void* dW1, void* dW2, int64_t M, int64_t D, int64_t H, int64_t Dout,
                             void* workspace, size_t workspace_bytes, void* stream) {
    return bwd_impl(x, W1, W2, preact, dy, dx, dW1, dW2, M, D, H, Dout, workspace, workspace_bytes, stream, false);
}

swiglu_status swiglu_mlp_bwd_residual(const void* x, const void* W1, const void* W2, const void* preact,
                                      const void* dy, void* dx, void* dW1, void* dW2, int64_t M, int64_t D,
                                      int64_t H, int64_t Dout, void* workspace, size_t workspace_bytes,
                                      void* stream) {
    if (D != Dout) return fail(SWIGLU_ERR_UNSUPPORTED_SHAPE, "residual block needs D == Dout");
    return bwd_impl(x, W1, W2, preact, dy, dx, dW1, dW2, M, D, H, Dout, workspace, workspace_bytes, stream, true);
}

swiglu_status swiglu_mlp_fused_grad_preact(const void* dy, const void* W2, const void* preact, void* grad_preact,
                                           void* h, int64_t M, int64_t H, int64_t Dout, void* stream) {
    if (M < 0 || H <= 0 || Dout <= 0) return fail(SWIGLU_ERR_INVALID_ARG, "swiglu_mlp_fused_grad_preact: a size is negative or zero");
    if (!dims_ok(H) || !dims_ok(Dout) || M >= (int64_t(1) << 31) || 2 * H >= (int64_t(1) << 31))
        return fail(SWIGLU_ERR_UNSUPPORTED_SHAPE, "swiglu_mlp_fused_grad_preact: unsupported shape (widths must be positive multiples of 8 below 2^31)");
    if (M == 0) return SWIGLU_OK;
    if (!dy || !W2 || !preact || !grad_preact || !h) return fail(SWIGLU_ERR_INVALID_ARG, "swiglu_mlp_fused_grad_preact: a required pointer is null");
    if (!aligned16(dy) || !aligned16(W2) || !aligned16(preact) || !aligned16(grad_preact) || !aligned16(h))
        return fail(SWIGLU_ERR_MISALIGNED, "swiglu_mlp_fused_grad_preact: a pointer is not 16-byte aligned");
    DeviceState* st;
    swiglu_status rc = get_device_state(&st);
    if (rc != SWIGLU_OK) return rc;
    return run_fused_bwd(st, dy, W2, preact, grad_preact, h, M, H, Dout, static_cast<cudaStream_t>(stream));
}

swiglu_status swiglu_mlp_gemm_bf16(const void* A, const void* B, void* Cp, int64_t M, int64_t N, int64_t K,
                                   int a_mn_major, int b_mn_major, void* stream) {
    if (M <= 0 || N <= 0 || K <= 0) return fail(SWIGLU_ERR_INVALID_ARG, "swiglu_mlp_gemm_bf16: a size is negative or zero");
    if (!A || !B || !Cp) return fail(SWIGLU_ERR_INVALID_ARG, "swiglu_mlp_gemm_bf16: a required pointer is null");
    const int64_t a_inner = a_mn_major ? M : K;
    const int64_t b_inner = b_mn_major ? N : K;
    if (a_inner % 8 || b_inner % 8 || N % 8 || M >= (int64_t(1) << 31) || N >= (int64_t(1) << 31) ||
        K >= (int64_t(1) << 31))
        return fail(SWIGLU_ERR_UNSUPPORTED_SHAPE, "swiglu_mlp_gemm_bf16: unsupported shape (widths must be positive multiples of 8 below 2^31)");
    if (!aligned16(A) || !aligned16(B) || !aligned16(Cp)) return fail(SWIGLU_ERR_MISALIGNED, "swiglu_mlp_gemm_bf16: a pointer is not 16-byte aligned");
    DeviceState* st;
    swiglu_status rc = get_device_state(&st);
    if (rc != SWIGLU_OK) return rc;
    return run_gemm(st, SWIGLU_KERNEL_GEMM, A, B, Cp, M, N, K, a_mn_major != 0, b_mn_major != 0,
                    static_cast<cudaStream_t>(stream));
}

swiglu_status swiglu_mlp_device_status(void* stream) {
    DeviceState* st;
    swiglu_status rc = get_device_state(&st);
    if (rc != SWIGLU_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return fail(SWIGLU_ERR_CUDA, "cudaStreamSynchronize", e);
    int word = 0;
    e = cudaMemcpy(&word, st->err_word, sizeof word, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return fail(SWIGLU_ERR_CUDA, "cudaMemcpy(error word)", e);
    if (word != 0) {
        const int zero = 0;
        e = cudaMemcpy(st->err_word, &zero, sizeof zero, cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return fail(SWIGLU_ERR_CUDA, "cudaMemcpy(error word)", e);
        std::snprintf(g_detail, sizeof g_detail, "device wait timed out (role bits 0x%x)", word);
        return SWIGLU_ERR_TIMEOUT;
    }
    return SWIGLU_OK;
}

const char* swiglu_mlp_strerror(swiglu_status status) {
    switch (status) {
        case SWIGLU_OK: return "SWIGLU_OK";
        case SWIGLU_ERR_INVALID_ARG: return "SWIGLU_ERR_INVALID_ARG: null pointer or invalid size";
        case SWIGLU_ERR_UNSUPPORTED_SHAPE: return "SWIGLU_ERR_UNSUPPORTED_SHAPE: D, H, Dout must be positive multiples of 8 below 2^31";
        case SWIGLU_ERR_MISALIGNED: return "SWIGLU_ERR_MISALIGNED: pointers must be 16-byte aligned";
        case SWIGLU_ERR_WORKSPACE_TOO_SMALL: return "SWIGLU_ERR_WORKSPACE_TOO_SMALL";
        case SWIGLU_ERR_LAUNCH: return "SWIGLU_ERR_LAUNCH: kernel launch or tensor-map encode failed";
        case SWIGLU_ERR_TIMEOUT: return "SWIGLU_ERR_TIMEOUT: a device-side wait ran out";
        case SWIGLU_ERR_CUDA: return "SWIGLU_ERR_CUDA: CUDA runtime error";
    }
    return "unknown swiglu_status";
}

const char* swiglu_mlp_last_error_detail(void) { return g_detail; }

void swiglu_mlp_set_wait_timeout_ns(uint64_t ns) { g_timeout_ns.store(ns ? ns : 1); }

void swiglu_mlp_set_debug_flags(int flags) { g_debug_flags.store(flags); }

void swiglu_mlp_set_raster_band(int n_tiles) { g_raster_band.store(n_tiles > 0 ? n_tiles : 0); }

int swiglu_mlp_split_plan(int64_t M, int64_t N, int64_t K, int units, int32_t* out, int cap) {
    if (M <= 0 || N <= 0 || K <= 0 || M >= (int64_t(1) << 31) || N >= (int64_t(1) << 31) || K >= (int64_t(1) << 31))
        return -1;
    if (split_ws_bytes(M, N, K) == 0) return -1;
    static thread_local ScheduledArgs a;
    std::memset(static_cast<KernelArgs*>(&a), 0, sizeof(KernelArgs));
    a.prob[0] = make_problem(M, N, K, (N + 2 * BN - 1) / (2 * BN), false, false, 2, 2);
    a.num_problems = 1;
    if (plan_split(a, units) < 0) return -1;
    int rows = 0;
    for (int u = 0; u < units; ++u) {
        for (int it = a.sched_off[u]; it < a.sched_off[u + 1]; ++it, ++rows) {
            if (!out || rows >= cap) continue;
            const int raw = a.sched[it];
            int32_t* r = out + 5 * rows;
            r[0] = u;
            r[1] = raw & SCHED_TILE_MASK;
            if (raw & SCHED_PIECE) {
                const SplitPiece& sp = a.split[u][(raw & SCHED_PIECE_PREFIX) ? 1 : 0];
                r[2] = sp.kb0;
                r[3] = sp.kb1;
                r[4] = sp.id;
            } else {
                r[2] = 0;
                r[3] = a.prob[0].k_blocks;
                r[4] = -1;
            }
        }
    }
    return rows;
}

void swiglu_mlp_trace_begin(void** events, int* kinds, int capacity) {
    Trace& tr = g_trace;
    const bool on = events && kinds && capacity > 0;
    tr.events = on ? reinterpret_cast<cudaEvent_t*>(events) : nullptr;
    tr.kinds = on ? kinds : nullptr;
    tr.capacity = on ? capacity : 0;
    tr.count = 0;
}

int swiglu_mlp_trace_end(void) {
    Trace& tr = g_trace;
    const int n = tr.count;
    tr = Trace();
    return n;
}

int swiglu_mlp_abi_version(void) { return 201; }

// ---------------------------------------------------------------- tensor-parallel shards
//
// "Lesson 24: MLP, GEMM and operator fusion in the Transformer", section 33: the first
// projection is split by columns (rank r keeps the hidden units J = [j0, j0 + Hs), i.e.
// W1 rows J and H + J, so that its SwiGLU is local) and the down projection by rows (W2
// columns J); each rank's y and dx are partial sums that the ranks add up (section 39:
// the reduction of one row chunk overlaps the GEMM of the next).

static swiglu_status shard_check(const char* who, int64_t D, int64_t H, int64_t Dout, int64_t j0, int64_t Hs) {
    if (!dims_ok(D) || !dims_ok(H) || !dims_ok(Dout) || !dims_ok(Hs) || j0 < 0 || j0 % 8 != 0 || j0 + Hs > H) {
        std::snprintf(g_detail, sizeof g_detail,
                      "%s: need D, H, Dout, Hs positive multiples of 8 and 0 <= j0 (a multiple of 8), j0 + Hs <= H", who);
        return SWIGLU_ERR_UNSUPPORTED_SHAPE;
    }
    return SWIGLU_OK;
}

swiglu_status swiglu_mlp_tp_shard_pack(const void* W1, const void* W2, void* W1_shard, void* W2_shard, int64_t D,
                                       int64_t H, int64_t Dout, int64_t j0, int64_t Hs, void* stream) {
    swiglu_status rc = shard_check("swiglu_mlp_tp_shard_pack", D, H, Dout, j0, Hs);
    if (rc != SWIGLU_OK) return rc;
    if (!W1 || !W2 || !W1_shard || !W2_shard) return fail(SWIGLU_ERR_INVALID_ARG, "swiglu_mlp_tp_shard_pack: a required pointer is null");
    if (!aligned16(W1) || !aligned16(W2) || !aligned16(W1_shard) || !aligned16(W2_shard))
        return fail(SWIGLU_ERR_MISALIGNED, "swiglu_mlp_tp_shard_pack: a pointer is not 16-byte aligned");
    DeviceState* st;
    rc = get_device_state(&st);
    if (rc != SWIGLU_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const uint8_t* w1 = static_cast<const uint8_t*>(W1);
    uint8_t* w1s = static_cast<uint8_t*>(W1_shard);
    const size_t block = (size_t)Hs * D * 2;   // Hs rows of W1
    cudaError_t e = cudaMemcpyAsync(w1s, w1 + (size_t)j0 * D * 2, block, cudaMemcpyDeviceToDevice, s);   // left rows J
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(w1s + block, w1 + (size_t)(H + j0) * D * 2, block, cudaMemcpyDeviceToDevice, s);   // gate rows H + J
    if (e == cudaSuccess)   // W2 columns J: Dout rows of Hs values, source pitch H
        e = cudaMemcpy2DAsync(W2_shard, (size_t)Hs * 2, static_cast<const uint8_t*>(W2) + (size_t)j0 * 2, (size_t)H * 2,
                              (size_t)Hs * 2, (size_t)Dout, cudaMemcpyDeviceToDevice, s);
    return e == cudaSuccess ? SWIGLU_OK : fail(SWIGLU_ERR_CUDA, "swiglu_mlp_tp_shard_pack: copy", e);
}

swiglu_status swiglu_mlp_tp_shard_unpack_grads(const void* dW1_shard, const void* dW2_shard, void* dW1, void* dW2,
                                               int64_t D, int64_t H, int64_t Dout, int64_t j0, int64_t Hs,
                                               void* stream) {
    swiglu_status rc = shard_check("swiglu_mlp_tp_shard_unpack_grads", D, H, Dout, j0, Hs);
    if (rc != SWIGLU_OK) return rc;
    if (!dW1 || !dW2 || !dW1_shard || !dW2_shard)
        return fail(SWIGLU_ERR_INVALID_ARG, "swiglu_mlp_tp_shard_unpack_grads: a required pointer is null");
    if (!aligned16(dW1) || !aligned16(dW2) || !aligned16(dW1_shard) || !aligned16(dW2_shard))
        return fail(SWIGLU_ERR_MISALIGNED, "swiglu_mlp_tp_shard_unpack_grads: a pointer is not 16-byte aligned");
    DeviceState* st;
    rc = get_device_state(&st);
    if (rc != SWIGLU_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const uint8_t* g1s = static_cast<const uint8_t*>(dW1_shard);
    uint8_t* g1 = static_cast<uint8_t*>(dW1);
    const size_t block = (size_t)Hs * D * 2;
    cudaError_t e = cudaMemcpyAsync(g1 + (size_t)j0 * D * 2, g1s, block, cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(g1 + (size_t)(H + j0) * D * 2, g1s + block, block, cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess)
        e = cudaMemcpy2DAsync(static_cast<uint8_t*>(dW2) + (size_t)j0 * 2, (size_t)H * 2, dW2_shard, (size_t)Hs * 2,
                              (size_t)Hs * 2, (size_t)Dout, cudaMemcpyDeviceToDevice, s);
    return e == cudaSuccess ? SWIGLU_OK : fail(SWIGLU_ERR_CUDA, "swiglu_mlp_tp_shard_unpack_grads: copy", e);
}

swiglu_status swiglu_mlp_tp_fwd(const void* x, const void* W1_shard, const void* W2_shard, void* preact_shard,
                                void* y_partial, int64_t M, int64_t D, int64_t Hs, int64_t Dout, int n_chunks,
                                void* const* chunk_events, void* workspace, size_t workspace_bytes, void* stream) {
    if (n_chunks < 1 || n_chunks > 1024) return fail(SWIGLU_ERR_INVALID_ARG, "swiglu_mlp_tp_fwd: n_chunks must be in 1..1024");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    auto record_from = [&](int c0) -> swiglu_status {
        for (int c = c0; chunk_events && c < n_chunks; ++c) {
            const swiglu_status r = record_event(chunk_events[c], s);
            if (r != SWIGLU_OK) return r;
        }
        return SWIGLU_OK;
    };
    if (M <= 0 || n_chunks == 1 || use_skinny(M)) {
        // one piece: the block forward on the shard, every chunk ready at its end
        const swiglu_status rc = fwd_impl(x, W1_shard, W2_shard, preact_shard, y_partial, M, D, Hs, Dout, workspace,
                                          workspace_bytes, stream, false);
        return rc != SWIGLU_OK ? rc : record_from(0);
    }
    // the same argument checks as the forward
    swiglu_status rc = fwd_impl(x, W1_shard, W2_shard, preact_shard, y_partial, 0, D, Hs, Dout, workspace,
                                workspace_bytes, stream, false);
    if (rc != SWIGLU_OK) return rc;
    if (!x || !W1_shard || !W2_shard || !preact_shard || !y_partial || !workspace)
        return fail(SWIGLU_ERR_INVALID_ARG, "swiglu_mlp_tp_fwd: a required pointer is null");
    if (!aligned16(x) || !aligned16(W1_shard) || !aligned16(W2_shard) || !aligned16(preact_shard) ||
        !aligned16(y_partial) || !aligned16(workspace))
        return fail(SWIGLU_ERR_MISALIGNED, "swiglu_mlp_tp_fwd: a pointer is not 16-byte aligned");
    if (M >= (int64_t(1) << 31)) return fail(SWIGLU_ERR_UNSUPPORTED_SHAPE, "swiglu_mlp_tp_fwd: M too large");
    if (workspace_bytes < swiglu_mlp_fwd_workspace_size(M, D, Hs, Dout))
        return fail(SWIGLU_ERR_WORKSPACE_TOO_SMALL, "swiglu_mlp_tp_fwd: workspace smaller than the size query returns");
    DeviceState* st;
    rc = get_device_state(&st);
    if (rc != SWIGLU_OK) return rc;
    uint8_t* h = static_cast<uint8_t*>(workspace);
    rc = run_fwd_preact(st, x, W1_shard, preact_shard, h, M, D, Hs, s);   // every row: preact and h of the shard
    if (rc != SWIGLU_OK) return rc;
    // the down projection in row chunks of whole 256-row tiles; chunk c's partial y is
    // complete when chunk_events[c] fires.  Chunks alternate between the caller's stream and
    // a second stream of this thread, so that each chunk's CTA pairs start on the SMs the
    // previous chunk's last round leaves idle (one launch per chunk would otherwise end in a
    // part-empty round each); the caller's stream waits for the second one at the end.
    cudaStream_t side;
    cudaEvent_t fork, join;
    rc = side_stream(&side, &fork, &join);
    if (rc != SWIGLU_OK) return rc;
    cudaError_t e = cudaEventRecord(fork, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(side, fork, 0);
    if (e != cudaSuccess) return fail(SWIGLU_ERR_CUDA, "swiglu_mlp_tp_fwd: fork onto the second stream", e);
    const int64_t per = ((M + n_chunks - 1) / n_chunks + 2 * BM - 1) / (2 * BM) * (2 * BM);
    for (int c = 0; c < n_chunks; ++c) {
        cudaStream_t sc = (c & 1) ? side : s;
        const int64_t r0 = (int64_t)c * per;
        if (r0 < M) {
            const int64_t rows = std::min<int64_t>(per, M - r0);
            rc = run_gemm(st, SWIGLU_KERNEL_FWD_DOWN, h + (size_t)r0 * Hs * 2, W2_shard,
                          static_cast<uint8_t*>(y_partial) + (size_t)r0 * Dout * 2, rows, Dout, Hs, false, false, sc);
            if (rc != SWIGLU_OK) return rc;
        }
        if (chunk_events) {
            rc = record_event(chunk_events[c], sc);
            if (rc != SWIGLU_OK) return rc;
        }
    }
    e = cudaEventRecord(join, side);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, join, 0);
    if (e != cudaSuccess) return fail(SWIGLU_ERR_CUDA, "swiglu_mlp_tp_fwd: join the second stream", e);
    return SWIGLU_OK;
}

swiglu_status swiglu_mlp_tp_bwd(const void* x, const void* W1_shard, const void* W2_shard, const void* preact_shard,
                                const void* dy, void* dx_partial, void* dW1_shard, void* dW2_shard, int64_t M,
                                int64_t D, int64_t Hs, int64_t Dout, void* dx_event, void* workspace,
                                size_t workspace_bytes, void* stream) {
    return bwd_impl(x, W1_shard, W2_shard, preact_shard, dy, dx_partial, dW1_shard, dW2_shard, M, D, Hs, Dout,
                    workspace, workspace_bytes, stream, false, dx_event);
}

int64_t swiglu_mlp_tp_chunk_rows(int64_t M, int n_chunks) {
    if (M <= 0 || n_chunks < 1) return 0;
    if (n_chunks == 1 || use_skinny(M)) return M;
    return ((M + n_chunks - 1) / n_chunks + 2 * BM - 1) / (2 * BM) * (2 * BM);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free forward.
//
// Some callers cannot hand the library a workspace: a plugin whose host
// framework owns every device allocation and exposes no scratch hook, a
// real-time loop that must not call cudaMalloc (it can synchronise the device),
// or a process whose device memory budget is fixed at start-up.  For them the
// forward's transient h lives in a fixed array in this library's own device
// memory.  The array exists on every GPU that loads the library, for the life
// of the process.
// ---------------------------------------------------------------------------
namespace swiglu {
namespace {

__device__ __align__(256) uint8_t g_fwd_scratch[SWIGLU_MLP_NOALLOC_SCRATCH_BYTES];

std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices];

// Device address of g_fwd_scratch on the current device, looked up once per device
// (the host-side name of the array is not a device address).
swiglu_status scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) return fail(SWIGLU_ERR_CUDA, "cudaGetDevice", e);
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_fwd_scratch);
        if (e != cudaSuccess || !p) return fail(SWIGLU_ERR_CUDA, "cudaGetSymbolAddress(static scratch)", e);
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return SWIGLU_OK;
}

}  // namespace
}  // namespace swiglu

extern "C" swiglu_status swiglu_mlp_fwd_noalloc(const void* x, const void* W1, const void* W2, void* preact,
                                                void* y, int64_t M, int64_t D, int64_t H, int64_t Dout,
                                                void* stream) {
    if (M < 0 || D <= 0 || H <= 0 || Dout <= 0) return fail(SWIGLU_ERR_INVALID_ARG, "swiglu_mlp_fwd_noalloc: a size is negative or zero");
    if (!dims_ok(D) || !dims_ok(H) || !dims_ok(Dout) || M >= (int64_t(1) << 31) || 2 * H >= (int64_t(1) << 31))
        return fail(SWIGLU_ERR_UNSUPPORTED_SHAPE, "swiglu_mlp_fwd_noalloc: unsupported shape (widths must be positive multiples of 8 below 2^31)");
    if (M == 0) return SWIGLU_OK;
    if (!x || !W1 || !W2 || !preact || !y) return fail(SWIGLU_ERR_INVALID_ARG, "swiglu_mlp_fwd_noalloc: a required pointer is null");
    if (!aligned16(x) || !aligned16(W1) || !aligned16(W2) || !aligned16(preact) || !aligned16(y))
        return fail(SWIGLU_ERR_MISALIGNED, "swiglu_mlp_fwd_noalloc: a pointer is not 16-byte aligned");
    const size_t need = (size_t)M * (size_t)H * 2;
    if (need > (size_t)SWIGLU_MLP_NOALLOC_SCRATCH_BYTES) {
        std::snprintf(g_detail, sizeof g_detail,
                      "swiglu_mlp_fwd_noalloc: h needs %zu bytes (M*H*2) but the built-in scratch holds %zu",
                      need, (size_t)SWIGLU_MLP_NOALLOC_SCRATCH_BYTES);
        return SWIGLU_ERR_WORKSPACE_TOO_SMALL;
    }
    DeviceState* st;
    swiglu_status rc = get_device_state(&st);
    if (rc != SWIGLU_OK) return rc;
    void* h = nullptr;
    rc = scratch_address(&h);
    if (rc != SWIGLU_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    rc = run_fwd_preact(st, x, W1, preact, h, M, D, H, s);
    if (rc != SWIGLU_OK) return rc;
    return run_gemm(st, SWIGLU_KERNEL_FWD_DOWN, h, W2, y, M, Dout, H, false, false, s);
}

// ---------------------------------------------------------------------------
// Mixture of experts ("Lesson 24: MLP, GEMM and operator fusion in the
// Transformer", sections 41-43): every expert is a SwiGLU block of its own and
// receives its own number of tokens.  Each step of the block runs as ONE
// persistent launch over all experts' GEMMs (a grouped GEMM): the launch reads a
// table of problems -- per expert its tensor maps, clipped to that expert's
// rows, and sizes -- from global memory, and the clusters walk a host tile list
// that balances the experts' tiles longest-first.
// ---------------------------------------------------------------------------
namespace swiglu {
namespace {

constexpr int kMaxUnits = 1024;          // bound on the clusters of one launch (table sizing)
constexpr int kStageSlots = 8;

// Pinned host slots the problem tables are copied from (a pageable source could
// make cudaMemcpyAsync wait for the stream).  A slot is refilled only after the
// copy enqueued from it kStageSlots tables earlier has completed.
struct Staging {
    uint8_t* host = nullptr;
    size_t cap = 0;
    cudaEvent_t done = nullptr;
};
std::mutex g_stage_mutex;
Staging g_stage[kMaxDevices][kStageSlots];
int g_stage_next[kMaxDevices];

swiglu_status stage_copy(void* dst, const std::vector<uint8_t>& img, cudaStream_t s) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(SWIGLU_ERR_CUDA, "cudaGetDevice", e);
    std::lock_guard<std::mutex> lock(g_stage_mutex);
    Staging& sl = g_stage[dev][g_stage_next[dev]];
    g_stage_next[dev] = (g_stage_next[dev] + 1) % kStageSlots;
    if (sl.done) {
        e = cudaEventSynchronize(sl.done);
        if (e != cudaSuccess) return fail(SWIGLU_ERR_CUDA, "cudaEventSynchronize(table staging)", e);
    } else {
        e = cudaEventCreateWithFlags(&sl.done, cudaEventDisableTiming);
        if (e != cudaSuccess) return fail(SWIGLU_ERR_CUDA, "cudaEventCreate(table staging)", e);
    }
    if (sl.cap < img.size()) {
        if (sl.host) cudaFreeHost(sl.host);
        sl.host = nullptr;
        sl.cap = 0;
        const size_t cap = std::max(img.size(), size_t(1) << 18);
        e = cudaHostAlloc(reinterpret_cast<void**>(&sl.host), cap, cudaHostAllocDefault);
        if (e != cudaSuccess) return fail(SWIGLU_ERR_CUDA, "cudaHostAlloc(table staging)", e);
        sl.cap = cap;
    }
    std::memcpy(sl.host, img.data(), img.size());
    e = cudaMemcpyAsync(dst, sl.host, img.size(), cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return fail(SWIGLU_ERR_CUDA, "cudaMemcpyAsync(problem table)", e);
    e = cudaEventRecord(sl.done, s);
    if (e != cudaSuccess) return fail(SWIGLU_ERR_CUDA, "cudaEventRecord(table staging)", e);
    return SWIGLU_OK;
}

// Device bytes of one launch's table: entries, cluster offsets, tile list, and
// slack to start the entries on a 256-byte boundary (tensor maps in global memory
// must be 64-byte aligned; the workspace is only 16-byte aligned).
size_t table_bytes(size_t entries, size_t tiles) {
    return 256 + round256(entries * sizeof(TableEntry)) + round256((kMaxUnits + 1) * sizeof(int)) +
           round256(tiles * sizeof(int));
}

// One launch over the problems in `ents` (tensor maps and problems filled in),
// its table written to dev_table (dev_bytes available) in stream order.
template <int EPI, int CG>
swiglu_status launch_table(DeviceState* st, int kind, std::vector<TableEntry>& ents, void* dev_table,
                           size_t dev_bytes, cudaStream_t s) {
    const int n = (int)ents.size();
    if (n == 0) return SWIGLU_OK;
    if (n >= (1 << (31 - TABLE_TILE_BITS))) return fail(SWIGLU_ERR_UNSUPPORTED_SHAPE, "too many problems");
    long long tiles = 0;
    for (TableEntry& e : ents) {
        const long long t = (long long)e.prob.tiles_m * e.prob.tiles_n;
        if (t >= (1 << TABLE_TILE_BITS)) return fail(SWIGLU_ERR_UNSUPPORTED_SHAPE, "too many tiles in one problem");
        e.prob.tile_begin = (int)tiles;
        tiles += t;
    }
    if (tiles == 0) return SWIGLU_OK;
    if (table_bytes((size_t)n, (size_t)tiles) > dev_bytes) return fail(SWIGLU_ERR_WORKSPACE_TOO_SMALL, "problem table");
    const uintptr_t raw = reinterpret_cast<uintptr_t>(dev_table);
    dev_table = reinterpret_cast<void*>((raw + 255) & ~uintptr_t(255));
    // experts of one GEMM share k-blocks and operand layout: the kernel then takes them
    // from its parameters (a faster producer mainloop)
    bool common = true;
    for (const TableEntry& e : ents)
        common = common && e.prob.k_blocks == ents[0].prob.k_blocks && e.prob.a_mn == ents[0].prob.a_mn &&
                 e.prob.b_mn == ents[0].prob.b_mn && e.prob.a3d == ents[0].prob.a3d &&
                 e.prob.b3d == ents[0].prob.b3d;
    const int slots = common ? cluster_slots<EPI, CG, SRC_TABLE_COMMON>(st) : cluster_slots<EPI, CG, SRC_TABLE>(st);
    if (slots <= 0) return fail(SWIGLU_ERR_LAUNCH, "cudaOccupancyMaxActiveClusters");
    const int units = (int)std::min<long long>(tiles, std::min(slots, kMaxUnits));

    // longest-processing-time: problems by decreasing tile time, each tile to the least-loaded
    // cluster (a tile costs its mainloop plus one k-block time per accumulator slot for its epilogue)
    auto cost = [&](const Problem& p) { return tile_cost(p) + p.slots; };
    std::vector<int> order(n);
    for (int i = 0; i < n; ++i) order[i] = i;
    std::stable_sort(order.begin(), order.end(),
                     [&](int a, int b) { return cost(ents[a].prob) > cost(ents[b].prob); });
    std::vector<std::vector<int>> lists(units);
    using Slot = std::pair<double, int>;
    std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> heap;
    for (int u = 0; u < units; ++u) heap.push({0.0, u});
    for (int pi : order) {
        const Problem& p = ents[pi].prob;
        const int nt = p.tiles_m * p.tiles_n;
        for (int t = 0; t < nt; ++t) {
            Slot sl = heap.top();
            heap.pop();
            lists[sl.second].push_back((pi << TABLE_TILE_BITS) | t);
            heap.push({sl.first + cost(p), sl.second});
        }
    }
    const size_t off_sched_off = round256((size_t)n * sizeof(TableEntry));
    const size_t off_sched = off_sched_off + round256((kMaxUnits + 1) * sizeof(int));
    std::vector<uint8_t> img(off_sched + (size_t)tiles * sizeof(int));
    std::memcpy(img.data(), ents.data(), (size_t)n * sizeof(TableEntry));
    int* so = reinterpret_cast<int*>(img.data() + off_sched_off);
    int* sc = reinterpret_cast<int*>(img.data() + off_sched);
    int pos = 0;
    for (int u = 0; u < units; ++u) {
        so[u] = pos;
        for (int v : lists[u]) sc[pos++] = v;
    }
    so[units] = pos;
    swiglu_status rc = stage_copy(dev_table, img, s);
    if (rc != SWIGLU_OK) return rc;

    TableArgs a;
    std::memset(&a, 0, sizeof a);
    uint8_t* d = static_cast<uint8_t*>(dev_table);
    a.table = reinterpret_cast<const TableEntry*>(d);
    a.sched_off = reinterpret_cast<const int*>(d + off_sched_off);
    a.sched = reinterpret_cast<const int*>(d + off_sched);
    a.num_problems = n;
    a.num_tiles = (int)tiles;
    a.timeout_ns = g_timeout_ns.load();
    a.err = st->err_word;
    a.debug_flags = g_debug_flags.load();
    a.common_k_blocks = ents[0].prob.k_blocks;
    a.common_a_mn = ents[0].prob.a_mn;
    a.common_b_mn = ents[0].prob.b_mn;
    a.common_a3d = ents[0].prob.a3d;
    a.common_b3d = ents[0].prob.b3d;
    if (common) return launch_grid<EPI, CG, SRC_TABLE_COMMON>(st, kind, a, units, s);
    return launch_grid<EPI, CG, SRC_TABLE>(st, kind, a, units, s);
}

// Expert segments: off[e] .. off[e + 1] are expert e's rows.
bool moe_offsets(const int64_t* counts, int64_t E, std::vector<int64_t>& off) {
    if (!counts || E <= 0 || E > 682) return false;   // 3E problems of one launch fit the table's index bits
    off.assign((size_t)E + 1, 0);
    for (int64_t e = 0; e < E; ++e) {
        if (counts[e] < 0 || counts[e] >= (int64_t(1) << 31)) return false;
        off[e + 1] = off[e] + counts[e];
    }
    return off[E] < (int64_t(1) << 31);
}

// Row tiles of one expert: 256-row CTA-pair tiles unless they would compute 25 %
// more padded rows than 128-row tiles over all experts (very many small experts).
// The pair kernels' deeper operand ring and halved B traffic outweigh moderate
// padding: with 64 experts of ~384 rows (17 % more rows) pairs measured 3.5 % faster.
// Host-only test hook bit: MoE launches keep CTA pairs whatever the padding.
constexpr int DEBUG_MOE_PAIRS = 16;

int moe_pick_cg(const std::vector<int64_t>& off) {
    if (g_debug_flags.load() & DEBUG_FORCE_SINGLE_CTA) return 1;
    if (g_debug_flags.load() & DEBUG_MOE_PAIRS) return 2;
    long long pad2 = 0, pad1 = 0;
    for (size_t e = 0; e + 1 < off.size(); ++e) {
        const long long m = off[e + 1] - off[e];
        pad2 += (m + 2 * BM - 1) / (2 * BM) * (2 * BM);
        pad1 += (m + BM - 1) / BM * BM;
    }
    return pad2 * 100 <= pad1 * 125 ? 2 : 1;
}

// Tile counts for the workspace bound (128-row tiles: never fewer than 256-row ones).
long long moe_row_tiles(const std::vector<int64_t>& off, int64_t n_tiles) {
    long long t = 0;
    for (size_t e = 0; e + 1 < off.size(); ++e) t += (off[e + 1] - off[e] + BM - 1) / BM * n_tiles;
    return t;
}

struct MoeDims {
    int64_t E, D, H, Dout, T;
};

size_t moe_fwd_tables(const std::vector<int64_t>& off, const MoeDims& d, size_t* first) {
    const size_t a = table_bytes((size_t)d.E, (size_t)moe_row_tiles(off, (d.H + BN / 2 - 1) / (BN / 2)));
    const size_t b = table_bytes((size_t)d.E, (size_t)moe_row_tiles(off, (d.Dout + BN - 1) / BN));
    if (first) *first = a;
    return a + b;
}

size_t moe_bwd_tables(const std::vector<int64_t>& off, const MoeDims& d, size_t* first) {
    const size_t a = table_bytes((size_t)d.E, (size_t)moe_row_tiles(off, (d.H + BN - 1) / BN));
    const long long dw_tiles = d.E * (((d.Dout + BM - 1) / BM) * ((d.H + BN - 1) / BN) +
                                      ((2 * d.H + BM - 1) / BM) * ((d.D + BN - 1) / BN));
    const size_t b = table_bytes((size_t)(3 * d.E), (size_t)(moe_row_tiles(off, (d.D + BN - 1) / BN) + dw_tiles));
    if (first) *first = a;
    return a + b;
}

// Plain-GEMM entry: C [M,N] = A * B^T, either operand K-major or MN-major.
// wide: 256 x 512 tiles (EPI_STORE_W launches).
bool fill_gemm(TableEntry& t, const GemmSpec& g, int cg, bool wide = false) {
    std::memset(&t, 0, sizeof t);
    bool a3d = false, b3d = false;
    if (!encode_operand(&t.a, g.A, g.M, g.K, g.a_mn, BM, &a3d)) return false;
    if (!encode_operand(&t.b, g.B, g.N, g.K, g.b_mn, BN / cg, &b3d)) return false;
    if (!encode_out_2d(&t.o0, g.C, g.M, g.N)) return false;
    const int64_t tile_n = wide ? 2 * BN : BN;
    t.prob = make_problem(g.M, g.N, g.K, (g.N + tile_n - 1) / tile_n, g.a_mn, g.b_mn, cg, wide ? 2 : 1);
    t.prob.a3d = a3d ? 1 : 0;
    t.prob.b3d = b3d ? 1 : 0;
    return true;
}

template <class T>
const T* at_row(const void* base, int64_t row, int64_t width) {
    return reinterpret_cast<const T*>(static_cast<const uint8_t*>(base) + row * width * 2);
}
template <class T>
T* at_row(void* base, int64_t row, int64_t width) {
    return reinterpret_cast<T*>(static_cast<uint8_t*>(base) + row * width * 2);
}

swiglu_status moe_check(const std::vector<int64_t>& off, const MoeDims& d) {
    if (!dims_ok(d.D) || !dims_ok(d.H) || !dims_ok(d.Dout) || 2 * d.H >= (int64_t(1) << 31))
        return fail(SWIGLU_ERR_UNSUPPORTED_SHAPE, "moe_check: unsupported shape (widths must be positive multiples of 8 below 2^31)");
    (void)off;
    return SWIGLU_OK;
}

}  // namespace
}  // namespace swiglu

extern "C" {

size_t swiglu_moe_fwd_workspace_size(const int64_t* counts, int64_t E, int64_t D, int64_t H, int64_t Dout) {
    std::vector<int64_t> off;
    if (!moe_offsets(counts, E, off) || H <= 0 || D <= 0 || Dout <= 0) return 0;
    const MoeDims d{E, D, H, Dout, off[E]};
    return round256((size_t)d.T * (size_t)H * 2) + moe_fwd_tables(off, d, nullptr);
}

size_t swiglu_moe_bwd_workspace_size(const int64_t* counts, int64_t E, int64_t D, int64_t H, int64_t Dout) {
    std::vector<int64_t> off;
    if (!moe_offsets(counts, E, off) || H <= 0 || D <= 0 || Dout <= 0) return 0;
    const MoeDims d{E, D, H, Dout, off[E]};
    return round256((size_t)d.T * (size_t)H * 2) + round256((size_t)d.T * (size_t)H * 4) +
           moe_bwd_tables(off, d, nullptr);
}

swiglu_status swiglu_moe_fwd(const void* x, const void* W1, const void* W2, void* preact, void* y,
                             const int64_t* counts, int64_t E, int64_t D, int64_t H, int64_t Dout,
                             void* workspace, size_t workspace_bytes, void* stream) {
    std::vector<int64_t> off;
    if (!moe_offsets(counts, E, off) || D <= 0 || H <= 0 || Dout <= 0) return fail(SWIGLU_ERR_INVALID_ARG, "swiglu_moe_fwd: invalid expert counts or a size that is not positive");
    const MoeDims d{E, D, H, Dout, off[E]};
    swiglu_status rc = moe_check(off, d);
    if (rc != SWIGLU_OK) return rc;
    if (d.T == 0) return SWIGLU_OK;
    if (!x || !W1 || !W2 || !preact || !y || !workspace) return fail(SWIGLU_ERR_INVALID_ARG, "swiglu_moe_fwd: a required pointer is null");
    if (!aligned16(x) || !aligned16(W1) || !aligned16(W2) || !aligned16(preact) || !aligned16(y) ||
        !aligned16(workspace))
        return fail(SWIGLU_ERR_MISALIGNED, "swiglu_moe_fwd: a pointer is not 16-byte aligned");
    if (workspace_bytes < swiglu_moe_fwd_workspace_size(counts, E, D, H, Dout))
        return fail(SWIGLU_ERR_WORKSPACE_TOO_SMALL, "swiglu_moe_fwd: workspace smaller than the size query returns");
    DeviceState* st;
    rc = get_device_state(&st);
    if (rc != SWIGLU_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* h = static_cast<uint8_t*>(workspace);
    size_t tab_a = 0;
    const size_t tabs = moe_fwd_tables(off, d, &tab_a);
    uint8_t* table_a = h + round256((size_t)d.T * (size_t)H * 2);
    uint8_t* table_b = table_a + tab_a;
    const int cg = moe_pick_cg(off);

    std::vector<TableEntry> ents;
    ents.reserve((size_t)E);
    for (int64_t e = 0; e < E; ++e) {        // preact_e = x_e @ W1[e]^T, SwiGLU epilogue
        const int64_t m = off[e + 1] - off[e];
        if (m == 0) continue;
        ents.emplace_back();
        TableEntry& t = ents.back();
        std::memset(&t, 0, sizeof t);
        const void* w1 = at_row<uint8_t>(W1, e * 2 * H, D);
        bool ok = encode_operand(&t.a, at_row<uint8_t>(x, off[e], D), m, D, false, BM);
        ok = ok && encode_3d(&t.b, w1, (uint64_t)D, (uint64_t)H, 2, (uint64_t)D * 2, (uint64_t)H * D * 2, 64,
                             BN / 2, 1, CU_TENSOR_MAP_SWIZZLE_128B);
        ok = ok && encode_paired(&t.o0, at_row<uint8_t>(preact, off[e], 2 * H), m, H, 32);
        ok = ok && encode_out_2d(&t.o1, at_row<uint8_t>(h, off[e], H), m, H);
        if (!ok) return fail(SWIGLU_ERR_LAUNCH, "tensor map encode (moe fwd_preact)");
        t.prob = make_problem(m, H, D, (H + BN / 2 - 1) / (BN / 2), false, false, cg);
    }
    rc = cg == 2 ? launch_table<EPI_SWIGLU_FWD, 2>(st, SWIGLU_KERNEL_FWD_PREACT, ents, table_a, tab_a, s)
                 : launch_table<EPI_SWIGLU_FWD, 1>(st, SWIGLU_KERNEL_FWD_PREACT, ents, table_a, tab_a, s);
    if (rc != SWIGLU_OK) return rc;
    std::vector<GemmSpec> specs;
    for (int64_t e = 0; e < E; ++e) {        // y_e = h_e @ W2[e]^T
        const int64_t m = off[e + 1] - off[e];
        if (m == 0) continue;
        specs.push_back(GemmSpec{at_row<uint8_t>(h, off[e], H), at_row<uint8_t>(W2, e * Dout, H),
                                 at_row<uint8_t>(y, off[e], Dout), m, Dout, H, false, false});
    }
    const bool wide = cg == 2 && wide_pays(st, specs.data(), (int)specs.size(), WIDE_LONG_K);
    ents.clear();
    for (const GemmSpec& g : specs) {
        ents.emplace_back();
        if (!fill_gemm(ents.back(), g, cg, wide)) return fail(SWIGLU_ERR_LAUNCH, "tensor map encode (moe fwd_down)");
    }
    if (wide) return launch_table<EPI_STORE_W, 2>(st, SWIGLU_KERNEL_FWD_DOWN, ents, table_b, tabs - tab_a, s);
    return cg == 2 ? launch_table<EPI_STORE, 2>(st, SWIGLU_KERNEL_FWD_DOWN, ents, table_b, tabs - tab_a, s)
                   : launch_table<EPI_STORE, 1>(st, SWIGLU_KERNEL_FWD_DOWN, ents, table_b, tabs - tab_a, s);
}

swiglu_status swiglu_moe_bwd(const void* x, const void* W1, const void* W2, const void* preact, const void* dy,
                             void* dx, void* dW1, void* dW2, const int64_t* counts, int64_t E, int64_t D,
                             int64_t H, int64_t Dout, void* workspace, size_t workspace_bytes, void* stream) {
    std::vector<int64_t> off;
    if (!moe_offsets(counts, E, off) || D <= 0 || H <= 0 || Dout <= 0) return fail(SWIGLU_ERR_INVALID_ARG, "swiglu_moe_bwd: invalid expert counts or a size that is not positive");
    const MoeDims d{E, D, H, Dout, off[E]};
    swiglu_status rc = moe_check(off, d);
    if (rc != SWIGLU_OK) return rc;
    if (!W1 || !W2 || !dW1 || !dW2) return fail(SWIGLU_ERR_INVALID_ARG, "swiglu_moe_bwd: a required pointer is null");
    if (!aligned16(W1) || !aligned16(W2) || !aligned16(dW1) || !aligned16(dW2)) return fail(SWIGLU_ERR_MISALIGNED, "swiglu_moe_bwd: a pointer is not 16-byte aligned");
    if (d.T > 0) {
        if (!x || !preact || !dy || !dx || !workspace) return fail(SWIGLU_ERR_INVALID_ARG, "swiglu_moe_bwd: a required pointer is null");
        if (!aligned16(x) || !aligned16(preact) || !aligned16(dy) || !aligned16(dx) || !aligned16(workspace))
            return fail(SWIGLU_ERR_MISALIGNED, "swiglu_moe_bwd: a pointer is not 16-byte aligned");
        if (workspace_bytes < swiglu_moe_bwd_workspace_size(counts, E, D, H, Dout))
            return fail(SWIGLU_ERR_WORKSPACE_TOO_SMALL, "swiglu_moe_bwd: workspace smaller than the size query returns");
    }
    DeviceState* st;
    rc = get_device_state(&st);
    if (rc != SWIGLU_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // experts without tokens: zero weight gradients
    for (int64_t e = 0; e < E; ++e) {
        if (off[e + 1] != off[e]) continue;
        cudaError_t ce = cudaMemsetAsync(at_row<uint8_t>(dW1, e * 2 * H, D), 0, (size_t)2 * H * D * 2, s);
        if (ce == cudaSuccess) ce = cudaMemsetAsync(at_row<uint8_t>(dW2, e * Dout, H), 0, (size_t)Dout * H * 2, s);
        if (ce != cudaSuccess) return fail(SWIGLU_ERR_CUDA, "cudaMemsetAsync(empty expert)", ce);
    }
    if (d.T == 0) return SWIGLU_OK;
    uint8_t* h = static_cast<uint8_t*>(workspace);
    uint8_t* gp = h + round256((size_t)d.T * (size_t)H * 2);
    size_t tab_a = 0;
    const size_t tabs = moe_bwd_tables(off, d, &tab_a);
    uint8_t* table_a = gp + round256((size_t)d.T * (size_t)H * 4);
    uint8_t* table_b = table_a + tab_a;
    const int cg = moe_pick_cg(off);

    std::vector<TableEntry> ents;
    ents.reserve((size_t)(3 * E));
    for (int64_t e = 0; e < E; ++e) {        // grad_h_e = dy_e @ W2[e] fused with the SwiGLU backward
        const int64_t m = off[e + 1] - off[e];
        if (m == 0) continue;
        ents.emplace_back();
        TableEntry& t = ents.back();
        std::memset(&t, 0, sizeof t);
        bool b3d = false;
        bool ok = encode_operand(&t.a, at_row<uint8_t>(dy, off[e], Dout), m, Dout, false, BM);
        ok = ok && encode_operand(&t.b, at_row<uint8_t>(W2, e * Dout, H), H, Dout, true, BN / cg, &b3d);
        ok = ok && encode_paired(&t.o0, at_row<uint8_t>(gp, off[e], 2 * H), m, H, 32, PRE_COLS);
        ok = ok && encode_out_2d(&t.o1, at_row<uint8_t>(h, off[e], H), m, H, PRE_COLS);
        ok = ok && encode_paired(&t.i0, at_row<uint8_t>(preact, off[e], 2 * H), m, H, 32, PRE_COLS);
        if (!ok) return fail(SWIGLU_ERR_LAUNCH, "tensor map encode (moe grad_h)");
        t.prob = make_problem(m, H, Dout, (H + BN - 1) / BN, false, true, cg);
        t.prob.b3d = b3d ? 1 : 0;
    }
    rc = cg == 2 ? launch_table<EPI_SWIGLU_BWD, 2>(st, SWIGLU_KERNEL_BWD_GRAD_H, ents, table_a, tab_a, s)
                 : launch_table<EPI_SWIGLU_BWD, 1>(st, SWIGLU_KERNEL_BWD_GRAD_H, ents, table_a, tab_a, s);
    if (rc != SWIGLU_OK) return rc;

    // dW2[e] = dy_e^T @ h_e, dx_e = grad_preact_e @ W1[e], dW1[e] = grad_preact_e^T @ x_e:
    // one launch over all experts (three with the ungrouped test hook)
    const int cgw = (g_debug_flags.load() & DEBUG_FORCE_SINGLE_CTA) ? 1 : 2;
    const bool grouped = !(g_debug_flags.load() & DEBUG_UNGROUPED);
    const int kinds[3] = {SWIGLU_KERNEL_BWD_DW2, SWIGLU_KERNEL_BWD_DX, SWIGLU_KERNEL_BWD_DW1};
    std::vector<GemmSpec> specs;
    for (int part = grouped ? -1 : 0; part < (grouped ? 0 : 3); ++part) {
        specs.clear();
        for (int64_t e = 0; e < E; ++e) {
            const int64_t m = off[e + 1] - off[e];
            if (m == 0) continue;
            const void* gpe = at_row<uint8_t>(gp, off[e], 2 * H);
            const GemmSpec g[3] = {
                {at_row<uint8_t>(dy, off[e], Dout), at_row<uint8_t>(h, off[e], H), at_row<uint8_t>(dW2, e * Dout, H),
                 Dout, H, m, true, true},
                {gpe, at_row<uint8_t>(W1, e * 2 * H, D), at_row<uint8_t>(dx, off[e], D), m, D, 2 * H, false, true},
                {gpe, at_row<uint8_t>(x, off[e], D), at_row<uint8_t>(dW1, e * 2 * H, D), 2 * H, D, m, true, true},
            };
            for (int q = 0; q < 3; ++q)
                if (part < 0 || q == part) specs.push_back(g[q]);
        }
        const bool wide = cgw == 2 && wide_pays(st, specs.data(), (int)specs.size(), WIDE_TABLE_GROUP);
        ents.clear();
        for (const GemmSpec& g : specs) {
            ents.emplace_back();
            if (!fill_gemm(ents.back(), g, cgw, wide)) return fail(SWIGLU_ERR_LAUNCH, "tensor map encode (moe bwd)");
        }
        const int kind = part < 0 ? SWIGLU_KERNEL_BWD_GEMMS : kinds[part];
        rc = wide ? launch_table<EPI_STORE_W, 2>(st, kind, ents, table_b, tabs - tab_a, s)
             : cgw == 2 ? launch_table<EPI_STORE, 2>(st, kind, ents, table_b, tabs - tab_a, s)
                        : launch_table<EPI_STORE, 1>(st, kind, ents, table_b, tabs - tab_a, s);
        if (rc != SWIGLU_OK) return rc;
    }
    return SWIGLU_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// FP8 forward ("Lesson 24: MLP, GEMM and operator fusion in the Transformer",
// section 26, the quantised GEMM epilogue; section 31, 8-bit weights): both
// products on FP8 E4M3 operands (tcgen05 kind::f8f6f4), fp32 accumulators, the
// first GEMM's epilogue scaling the accumulator, applying the SwiGLU and writing
// h quantised to E4M3; the second GEMM's epilogue scaling to bf16 y.
// ---------------------------------------------------------------------------
namespace swiglu {
namespace {

// Workspace of the FP8 forward: for M <= 64 the fp32 sums preact^T [2H, M16] and
// y^T [Dout, M16] (M16 = M rounded up to 16); nothing otherwise.
size_t fp8_fwd_ws(int64_t M, int64_t D, int64_t H, int64_t Dout, float** pt, float** yt, void* base) {
    if (!use_skinny(M)) return 0;
    const size_t a = round256(skinny_acc_bytes(2 * H, D, M, true));
    if (base) {
        *pt = static_cast<float*>(base);
        *yt = reinterpret_cast<float*>(static_cast<uint8_t*>(base) + a);
    }
    return a + round256(skinny_acc_bytes(Dout, H, M, true));
}

// M <= 64 tokens: weight-streaming FP8 products (transposed, split over K) and
// element-wise kernels that scale, apply the SwiGLU, quantise h and cast y.
swiglu_status run_fwd_fp8_skinny(DeviceState* st, const void* x8, const void* W1_8, const void* W2_8, float s_x,
                                 float s_w1, float s_w2, float s_h, void* preact, void* h8, void* y, int64_t M,
                                 int64_t D, int64_t H, int64_t Dout, void* ws, cudaStream_t s) {
    float *pt = nullptr, *yt = nullptr;
    fp8_fwd_ws(M, D, H, Dout, &pt, &yt, ws);
    Planes ptp, ytp;
    swiglu_status rc = run_skinny(st, SWIGLU_KERNEL_FWD_PREACT, W1_8, false, x8, pt, 2 * H, D, M, s, true, &ptp);
    if (rc != SWIGLU_OK) return rc;
    const int g = elementwise_grid(st, (long long)M * H);
    rc = launch_traced(SWIGLU_KERNEL_ELEMENTWISE, s, [&]() {
        skinny_swiglu_fwd_fp8_kernel<<<g, 256, 0, s>>>(ptp, s_x * s_w1, 1.0f / s_h,
                                                        static_cast<__nv_bfloat16*>(preact),
                                                        static_cast<uint8_t*>(h8), (int)M, (int)H);
        return cudaGetLastError();
    });
    if (rc != SWIGLU_OK) return rc;
    rc = run_skinny(st, SWIGLU_KERNEL_FWD_DOWN, W2_8, false, h8, yt, Dout, H, M, s, true, &ytp);
    if (rc != SWIGLU_OK) return rc;
    const int g2 = elementwise_grid(st, (long long)M * Dout);
    return launch_traced(SWIGLU_KERNEL_ELEMENTWISE, s, [&]() {
        skinny_cast_kernel<<<g2, 256, 0, s>>>(ytp, nullptr, static_cast<__nv_bfloat16*>(y), (int)M, (int)Dout,
                                              s_h * s_w2);
        return cudaGetLastError();
    });
}

swiglu_status run_fwd_fp8(DeviceState* st, const void* x8, const void* W1_8, const void* W2_8, float s_x,
                          float s_w1, float s_w2, float s_h, void* preact, void* h8, void* y, int64_t M,
                          int64_t D, int64_t H, int64_t Dout, void* ws, cudaStream_t s) {
    if (use_skinny(M))
        return run_fwd_fp8_skinny(st, x8, W1_8, W2_8, s_x, s_w1, s_w2, s_h, preact, h8, y, M, D, H, Dout, ws, s);
    constexpr CUtensorMapDataType U8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
    const int cg = pick_cg(M);
    KernelArgs a;
    std::memset(&a, 0, sizeof a);
    // x8 [M, D] and W1_8 [2H, D] as (k, j, half), 128 k values (bytes) per box row
    bool ok = encode_2d(&a.a[0], x8, (uint64_t)D, (uint64_t)M, (uint64_t)D, 2 * BK, BM, CU_TENSOR_MAP_SWIZZLE_128B, U8);
    ok = ok && encode_3d(&a.b[0], W1_8, (uint64_t)D, (uint64_t)H, 2, (uint64_t)D, (uint64_t)H * D, 2 * BK, BN / 2, 1,
                         CU_TENSOR_MAP_SWIZZLE_128B, U8);
    if (preact) ok = ok && encode_paired(&a.o0[0], preact, M, H, 32);
    // h8 [M, H]: 32-byte rows of this warp's 32 columns, unswizzled
    ok = ok && encode_2d(&a.o1, h8, (uint64_t)H, (uint64_t)M, (uint64_t)H, CHUNK, 32, CU_TENSOR_MAP_SWIZZLE_NONE, U8);
    if (!ok) return fail(SWIGLU_ERR_LAUNCH, "tensor map encode (fp8 fwd_preact)");
    a.num_problems = 1;
    a.prob[0] = make_problem(M, H, D, (H + BN / 2 - 1) / (BN / 2), false, false, cg);
    a.prob[0].k_blocks = (int)((D + 2 * BK - 1) / (2 * BK));
    a.prob[0].no_o0 = preact ? 0 : 1;
    a.scale_acc = s_x * s_w1;
    a.scale_out = 1.0f / s_h;
    swiglu_status rc = cg == 2
        ? launch<EPI_SWIGLU_FWD, 2, SRC_SINGLE, OP_E4M3>(st, SWIGLU_KERNEL_FWD_PREACT, a, s)
        : launch<EPI_SWIGLU_FWD, 1, SRC_SINGLE, OP_E4M3>(st, SWIGLU_KERNEL_FWD_PREACT, a, s);
    if (rc != SWIGLU_OK) return rc;

    // y = (s_h s_w2) * (h8 @ W2_8^T)
    KernelArgs b;
    std::memset(&b, 0, sizeof b);
    ok = encode_2d(&b.a[0], h8, (uint64_t)H, (uint64_t)M, (uint64_t)H, 2 * BK, BM, CU_TENSOR_MAP_SWIZZLE_128B, U8);
    ok = ok && encode_2d(&b.b[0], W2_8, (uint64_t)H, (uint64_t)Dout, (uint64_t)H, 2 * BK, BN / cg,
                         CU_TENSOR_MAP_SWIZZLE_128B, U8);
    ok = ok && encode_out_2d(&b.o0[0], y, M, Dout);
    if (!ok) return fail(SWIGLU_ERR_LAUNCH, "tensor map encode (fp8 fwd_down)");
    b.num_problems = 1;
    b.prob[0] = make_problem(M, Dout, H, (Dout + BN - 1) / BN, false, false, cg);
    b.prob[0].k_blocks = (int)((H + 2 * BK - 1) / (2 * BK));
    b.scale_acc = s_h * s_w2;
    return cg == 2 ? launch<EPI_STORE, 2, SRC_SINGLE, OP_E4M3>(st, SWIGLU_KERNEL_FWD_DOWN, b, s)
                   : launch<EPI_STORE, 1, SRC_SINGLE, OP_E4M3>(st, SWIGLU_KERNEL_FWD_DOWN, b, s);
}

}  // namespace
}  // namespace swiglu

extern "C" size_t swiglu_mlp_fwd_fp8_workspace_size(int64_t M, int64_t D, int64_t H, int64_t Dout) {
    (void)D;
    if (M <= 0 || H <= 0 || Dout <= 0) return 0;
    return fp8_fwd_ws(M, D, H, Dout, nullptr, nullptr, nullptr);
}

extern "C" swiglu_status swiglu_mlp_fwd_fp8(const void* x8, const void* W1_8, const void* W2_8, float s_x,
                                            float s_w1, float s_w2, float s_h, void* preact, void* h8, void* y,
                                            int64_t M, int64_t D, int64_t H, int64_t Dout, void* workspace,
                                            size_t workspace_bytes, void* stream) {
    if (M < 0 || D <= 0 || H <= 0 || Dout <= 0) return fail(SWIGLU_ERR_INVALID_ARG, "swiglu_mlp_fwd_fp8: a size is negative or zero");
    if (D % 16 || H % 16 || !dims_ok(Dout) || D >= (int64_t(1) << 31) || 2 * H >= (int64_t(1) << 31) ||
        M >= (int64_t(1) << 31))
        return fail(SWIGLU_ERR_UNSUPPORTED_SHAPE, "fp8 forward: D and H multiples of 16, Dout of 8");
    if (!(s_x > 0.0f) || !(s_w1 > 0.0f) || !(s_w2 > 0.0f) || !(s_h > 0.0f) || !std::isfinite(1.0f / s_h))
        return fail(SWIGLU_ERR_INVALID_ARG, "fp8 forward: scales must be positive and finite");
    if (M == 0) return SWIGLU_OK;
    if (!x8 || !W1_8 || !W2_8 || !h8 || !y) return fail(SWIGLU_ERR_INVALID_ARG, "swiglu_mlp_fwd_fp8: a required pointer is null");
    if (!aligned16(x8) || !aligned16(W1_8) || !aligned16(W2_8) || !aligned16(h8) || !aligned16(y) ||
        (preact && !aligned16(preact)) || (workspace && !aligned16(workspace)))
        return fail(SWIGLU_ERR_MISALIGNED, "swiglu_mlp_fwd_fp8: a pointer is not 16-byte aligned");
    const size_t need = swiglu_mlp_fwd_fp8_workspace_size(M, D, H, Dout);
    if (need > 0 && (!workspace || workspace_bytes < need)) return fail(SWIGLU_ERR_WORKSPACE_TOO_SMALL, "swiglu_mlp_fwd_fp8: workspace smaller than the size query returns");
    DeviceState* st;
    swiglu_status rc = get_device_state(&st);
    if (rc != SWIGLU_OK) return rc;
    return run_fwd_fp8(st, x8, W1_8, W2_8, s_x, s_w1, s_w2, s_h, preact, h8, y, M, D, H, Dout, workspace,
                       static_cast<cudaStream_t>(stream));
}
