// api.cu -- the C ABI declared in include/mxfp4.h: argument checks, the device gate, TMA
// descriptor set-up and kernel launches.  Nothing here allocates device memory or
// synchronizes, except mxfp4_last_device_error, whose job is to synchronize.
#include <cudaTypedefs.h>

#include <atomic>
#include <cstring>
#include <mutex>

#include "launch.h"
#include "launch_fp8.h"
#include "mxfp4.h"
#include "ptx.cuh"

namespace {

// Device error word: kernels OR a site bit into it when a bounded wait runs out.
__device__ uint32_t g_error_word;

constexpr int kMaxDevices = 64;
constexpr int64_t kMaxDim = (int64_t{1} << 31) - 512;  // keeps tile coordinates in int32
// Modelled cost of a CTA-pair K step (cycles of one cluster) and of a tile's accumulator
// hand-over, for the choice of tile width.
constexpr double kPairNarrowStepCost = 512.0;
constexpr double kPairWideStepCost = 768.0;
constexpr double kPairHandoverCost = 1500.0;
// Tile order of the pair kernel: problems of up to kPairGroupAllRows row tiles walk all of
// them fastest (the co-resident clusters cover every A row tile, each B column tile is read
// once); taller ones walk groups of kPairGroupM row tiles, so A streams once instead of once
// per column tile (measured on the Flux wgrad, M 21504: 187.9 -> 180.1 us for dgrad + wgrad;
// a grouped order on the 18-row-tile forward cost 5-7 %).
constexpr int32_t kPairGroupAllRows = 24;
constexpr int32_t kPairGroupM = 8;
std::atomic<int> g_tile_policy{MXFP4_TILES_AUTO};   // mxfp4_gemm_set_tile_policy

struct DeviceState {
    int state = 0;  // 0 unknown, 1 supported, 2 unsupported
    int sms = 0;
    uint32_t* err = nullptr;
};

std::mutex g_mutex;
DeviceState g_devices[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode_tiled = nullptr;

mxfp4_status device_ready(DeviceState** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MXFP4_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return MXFP4_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState& d = g_devices[dev];
    if (d.state == 0) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return MXFP4_ERR_CUDA;
        if (major != 10 || minor != 3) {
            d.state = 2;
        } else {
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return MXFP4_ERR_CUDA;
            if (g_encode_tiled == nullptr) {
                void* fn = nullptr;
                cudaDriverEntryPointQueryResult q;
                if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                                     &q) != cudaSuccess ||
                    q != cudaDriverEntryPointSuccess || fn == nullptr)
                    return MXFP4_ERR_CUDA;
                g_encode_tiled = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
            }
            d.err = static_cast<uint32_t*>(p);
            d.sms = sms;
            d.state = 1;
        }
    }
    if (d.state != 1) return MXFP4_ERR_UNSUPPORTED_DEVICE;
    *out = &d;
    return MXFP4_OK;
}

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int64_t pad128(int64_t n) { return cdiv(n, 128) * 128; }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool encode_2d(CUtensorMap* map, CUtensorMapDataType type, const void* base, uint64_t inner,
               uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
               CUtensorMapSwizzle swizzle) {
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode_tiled(map, type, 2, const_cast<void*>(base), dims, strides, box, estr,
                                CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Argument checks of one quantization task (no device needed).
mxfp4_status quantize_check(const void* x, int64_t M, int64_t K, int64_t ldx, const void* q_row,
                            const void* s_row, const void* q_col, const void* s_col, mxfp4_scale_layout layout,
                            bool dual) {
    if (x == nullptr || q_row == nullptr || s_row == nullptr) return MXFP4_ERR_INVALID_ARG;
    if (dual && (q_col == nullptr || s_col == nullptr)) return MXFP4_ERR_INVALID_ARG;
    if (M < 1 || K < 1 || M > kMaxDim || K > kMaxDim || ldx < K || ldx > kMaxDim) return MXFP4_ERR_INVALID_ARG;
    if (layout != MXFP4_SCALE_PLAIN && layout != MXFP4_SCALE_TC) return MXFP4_ERR_INVALID_ARG;
    if (!aligned16(x) || (ldx % 8) != 0 || !aligned16(q_row) || !aligned16(s_row)) return MXFP4_ERR_MISALIGNED;
    if (dual && (!aligned16(q_col) || !aligned16(s_col))) return MXFP4_ERR_MISALIGNED;
    return MXFP4_OK;
}

// Fills slot j of the batch (tensor map and arguments) for a checked task.
mxfp4_status quantize_task(const void* x, int64_t M, int64_t K, int64_t ldx, void* q_row, void* s_row,
                           void* q_col, void* s_col, mxfp4_scale_layout layout, DeviceState* dev,
                           mxfp4::QuantBatch* b, int j, int32_t flags = 0, uint32_t rht_signs = 0) {
    if (!encode_2d(&b->maps[j], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, static_cast<uint64_t>(K),
                   static_cast<uint64_t>(M), static_cast<uint64_t>(ldx) * 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B))
        return MXFP4_ERR_CUDA;
    mxfp4::QuantArgs& a = b->args[j];
    a.M = M;
    a.K = K;
    a.tiles_m = static_cast<int32_t>(cdiv(M, 128));
    a.tiles_k = static_cast<int32_t>(cdiv(K, 128));
    a.q_row = static_cast<uint8_t*>(q_row);
    a.s_row = static_cast<uint8_t*>(s_row);
    a.q_col = static_cast<uint8_t*>(q_col);
    a.s_col = static_cast<uint8_t*>(s_col);
    a.ldq_row = pad128(K) / 2;
    a.ldq_col = pad128(M) / 2;
    a.kb_row = pad128(K) / 32;
    a.kb_col = pad128(M) / 32;
    a.tc_layout = layout == MXFP4_SCALE_TC ? 1 : 0;
    a.seed = 0;
    a.block_2d = (flags & MXFP4_QUANT_2D_BLOCKS) ? 1 : 0;
    a.rht = (flags & MXFP4_QUANT_RHT_COL) ? 1 : 0;
    a.rht_signs = rht_signs & 0xFFFFu;
    a.err = dev->err;
    const int64_t before = j > 0 ? b->tile_end[j - 1] : 0;
    const int64_t end = before + static_cast<int64_t>(a.tiles_m) * a.tiles_k;
    if (end > (int64_t{1} << 31) - 1) return MXFP4_ERR_INVALID_ARG;
    b->tile_end[j] = static_cast<int32_t>(end);
    b->count = j + 1;
    return MXFP4_OK;
}

mxfp4_status launch_batch(const mxfp4::QuantBatch& b, bool dual, DeviceState* dev, cudaStream_t stream,
                          bool sr = false) {
    const int64_t tiles = b.tile_end[b.count - 1];
    const int64_t cap = static_cast<int64_t>(dev->sms) * mxfp4::quantize_ctas_per_sm(sr);
    const int grid = static_cast<int>(tiles < cap ? tiles : cap);
    return mxfp4::launch_quantize(b, dual, sr, grid, stream) == cudaSuccess ? MXFP4_OK : MXFP4_ERR_CUDA;
}

mxfp4_status quantize_common(const void* x, int64_t M, int64_t K, int64_t ldx, void* q_row, void* s_row,
                             void* q_col, void* s_col, mxfp4_scale_layout layout, bool dual,
                             cudaStream_t stream, bool sr = false, uint64_t seed = 0, int32_t flags = 0,
                             uint32_t rht_signs = 0) {
    mxfp4_status st = quantize_check(x, M, K, ldx, q_row, s_row, q_col, s_col, layout, dual);
    if (st != MXFP4_OK) return st;
    DeviceState* dev = nullptr;
    st = device_ready(&dev);
    if (st != MXFP4_OK) return st;
    mxfp4::QuantBatch b;
    std::memset(&b, 0, sizeof(b));
    st = quantize_task(x, M, K, ldx, q_row, s_row, q_col, s_col, layout, dev, &b, 0, flags, rht_signs);
    if (st != MXFP4_OK) return st;
    b.args[0].seed = seed;
    return launch_batch(b, dual, dev, stream, sr);
}

__global__ void selftest_wait_kernel(uint32_t* err, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mxfp4::mbar_init(mxfp4::smem_addr(&bar), 1);
        abort_flag = 0;
        mxfp4::fence_barrier_init();
    }
    __syncwarp();
    if (threadIdx.x == 0) {
        // Nothing ever arrives on `bar`, so phase 0 never completes: the wait must give up.
        mxfp4::mbar_wait(mxfp4::smem_addr(&bar), 0, err, mxfp4::kErrSelftest, &abort_flag, limit_ns);
    }
    __syncwarp();
}

// Argument checks of one GEMM (no device needed).
mxfp4_status gemm_check(const mxfp4_gemm_task& t) {
    if (!t.a_q || !t.a_s || !t.b_q || !t.b_s || !t.c) return MXFP4_ERR_INVALID_ARG;
    if (t.M < 1 || t.N < 1 || t.K < 1 || t.M > kMaxDim || t.N > kMaxDim || t.K > kMaxDim)
        return MXFP4_ERR_INVALID_ARG;
    if (t.ldc < t.N || t.ldc > kMaxDim) return MXFP4_ERR_INVALID_ARG;
    if (t.out_dtype != MXFP4_OUT_BF16 && t.out_dtype != MXFP4_OUT_F32) return MXFP4_ERR_INVALID_ARG;
    if (!aligned16(t.a_q) || !aligned16(t.a_s) || !aligned16(t.b_q) || !aligned16(t.b_s) || !aligned16(t.c) ||
        (t.bias != nullptr && !aligned16(t.bias)))
        return MXFP4_ERR_MISALIGNED;
    const int64_t tiles = cdiv(t.M, mxfp4::kGemmBM) * cdiv(t.N, mxfp4::kGemmBN);
    if (tiles > (int64_t{1} << 31) - 1) return MXFP4_ERR_INVALID_ARG;
    return MXFP4_OK;
}

// Kernel arguments and the A, B (box of b_rows rows) and C tensor maps of a checked GEMM.
// C goes out through TMA stores when its pitch allows a tensor map (a multiple of 16
// bytes; the base is 16-byte aligned by the checks); otherwise with plain stores.
mxfp4_status gemm_fill(const mxfp4_gemm_task& t, DeviceState* dev, mxfp4::GemmArgs* g, CUtensorMap* amap,
                       CUtensorMap* bmap, CUtensorMap* cmap, uint32_t b_rows) {
    const int64_t kp = pad128(t.K);
    if (!encode_2d(amap, CU_TENSOR_MAP_DATA_TYPE_UINT8, t.a_q, static_cast<uint64_t>(kp / 2),
                   static_cast<uint64_t>(t.M), static_cast<uint64_t>(kp / 2), 128, mxfp4::kGemmBM,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(bmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, t.b_q, static_cast<uint64_t>(kp / 2),
                   static_cast<uint64_t>(t.N), static_cast<uint64_t>(kp / 2), 128, b_rows,
                   CU_TENSOR_MAP_SWIZZLE_128B))
        return MXFP4_ERR_CUDA;
    const int64_t esize = t.out_dtype == MXFP4_OUT_F32 ? 4 : 2;
    std::memset(cmap, 0, sizeof(*cmap));
    const bool c_tma = (t.ldc * esize) % 16 == 0 &&
                       encode_2d(cmap, t.out_dtype == MXFP4_OUT_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                                                     : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                                 t.c, static_cast<uint64_t>(t.N), static_cast<uint64_t>(t.M),
                                 static_cast<uint64_t>(t.ldc * esize), static_cast<uint32_t>(64 / esize), 32,
                                 CU_TENSOR_MAP_SWIZZLE_64B);
    g->M = t.M;
    g->N = t.N;
    g->tiles_m = static_cast<int32_t>(cdiv(t.M, mxfp4::kGemmBM));
    g->tiles_n = static_cast<int32_t>(cdiv(t.N, mxfp4::kGemmBN));
    g->tiles_m2 = static_cast<int32_t>(cdiv(t.M, 256));
    g->k_stages = static_cast<int32_t>(cdiv(kp, 256));
    g->kb4 = static_cast<int32_t>(kp / 128);
    g->groups_b = static_cast<int32_t>(cdiv(t.N, 128));
    g->a_s = static_cast<const uint8_t*>(t.a_s);
    g->b_s = static_cast<const uint8_t*>(t.b_s);
    g->c = t.c;
    g->ldc = t.ldc;
    g->out_f32 = t.out_dtype == MXFP4_OUT_F32 ? 1 : 0;
    g->c_tma = c_tma ? 1 : 0;
    g->bias = static_cast<const uint16_t*>(t.bias);
    g->err = dev->err;
    return MXFP4_OK;
}

// Appends a checked GEMM to the CTA-pair batch (B box 128 rows, scale maps; wide tiles: the
// 64-row B map too, and three scale groups of B per box).
mxfp4_status gemm_fill_pair(const mxfp4_gemm_task& t, DeviceState* dev, mxfp4::GemmPairBatch* b, bool wide) {
    const int j = b->count;
    mxfp4::GemmArgs& g = b->args[j];
    mxfp4_status st = gemm_fill(t, dev, &g, &b->amap[j], &b->bmap[j], &b->cmap[j], 128);
    if (st != MXFP4_OK) return st;
    const int64_t kp = pad128(t.K);
    if (!encode_2d(&b->sfamap[j], CU_TENSOR_MAP_DATA_TYPE_UINT64, t.a_s, static_cast<uint64_t>(g.kb4) * 64,
                   static_cast<uint64_t>(cdiv(t.M, 128)), static_cast<uint64_t>(g.kb4) * 512, 128, 1,
                   CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_2d(&b->sfbmap[j], CU_TENSOR_MAP_DATA_TYPE_UINT64, t.b_s, static_cast<uint64_t>(g.kb4) * 64,
                   static_cast<uint64_t>(cdiv(t.N, 128)), static_cast<uint64_t>(g.kb4) * 512, 128, wide ? 3 : 2,
                   CU_TENSOR_MAP_SWIZZLE_NONE) ||
        (wide && !encode_2d(&b->bmap2[j], CU_TENSOR_MAP_DATA_TYPE_UINT8, t.b_q, static_cast<uint64_t>(kp / 2),
                            static_cast<uint64_t>(t.N), static_cast<uint64_t>(kp / 2), 128, 64,
                            CU_TENSOR_MAP_SWIZZLE_128B)))
        return MXFP4_ERR_CUDA;
    if (wide) {
        // C as bf16 {N, M}, box {32 columns, 128 rows}: a column group's four epilogue warps
        // store their 128 rows together
        if (!g.c_tma || g.out_f32 ||
            !encode_2d(&b->cmap[j], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, t.c, static_cast<uint64_t>(t.N),
                       static_cast<uint64_t>(t.M), static_cast<uint64_t>(t.ldc * 2), 32, 128, CU_TENSOR_MAP_SWIZZLE_64B))
            return MXFP4_ERR_INVALID_ARG;
        g.tiles_n = static_cast<int32_t>(cdiv(t.N, mxfp4::kPairTileNWide));
    }
    g.group_m = g.tiles_m2 <= kPairGroupAllRows ? g.tiles_m2 : kPairGroupM;
    const int64_t before = j > 0 ? b->tile_end[j - 1] : 0;
    const int64_t end = before + static_cast<int64_t>(g.tiles_m2) * g.tiles_n;
    if (end > (int64_t{1} << 31) - 1) return MXFP4_ERR_INVALID_ARG;
    b->tile_end[j] = static_cast<int32_t>(end);
    b->count = j + 1;
    return MXFP4_OK;
}

// Tile width of a CTA-pair launch.  Wide tiles (256 x 384) need every problem's output in
// bf16 through TMA stores.  Otherwise the launch takes the width with the lower modelled
// time: the tiles are dealt round-robin to the clusters, as the kernel walks them; a tile
// costs its K steps times its width (the MMA time, in units of 128 columns) times the
// width's measured efficiency, plus a fixed accumulator hand-over; the busiest cluster sets
// the time.
double pair_time_model(const mxfp4_gemm_task* tasks, const bool* on_pair, int count, int clusters, int tile_n) {
    if (clusters <= 0) return 1e300;
    const double per_step = (tile_n == mxfp4::kPairTileNWide ? kPairWideStepCost : kPairNarrowStepCost);
    double busiest = 0.0;
    // tiles of each problem occupy a contiguous range of launch tile indices
    int64_t begin[MXFP4_MAX_BATCH], ntiles[MXFP4_MAX_BATCH];
    double cost[MXFP4_MAX_BATCH];
    int64_t at = 0;
    int n = 0;
    for (int j = 0; j < count; ++j) {
        if (!on_pair[j]) continue;
        const int64_t kp = pad128(tasks[j].K);
        begin[n] = at;
        ntiles[n] = cdiv(tasks[j].M, 256) * cdiv(tasks[j].N, tile_n);
        cost[n] = static_cast<double>(cdiv(kp, 256)) * per_step + kPairHandoverCost;
        at += ntiles[n];
        ++n;
    }
    const int64_t used = at < clusters ? at : clusters;
    for (int64_t c = 0; c < used; ++c) {
        double sum = 0.0;
        for (int p = 0; p < n; ++p) {
            // launch tiles t in [begin, begin + ntiles) with t = c (mod clusters)
            const int64_t lo = begin[p], hi = begin[p] + ntiles[p];
            const int64_t first = lo + ((c - lo % clusters) % clusters + clusters) % clusters;
            if (first < hi) sum += static_cast<double>((hi - 1 - first) / clusters + 1) * cost[p];
        }
        busiest = sum > busiest ? sum : busiest;
    }
    return busiest;
}

bool pair_use_wide(const mxfp4_gemm_task* tasks, const bool* on_pair, int count, int narrow_clusters,
                   int wide_clusters) {
    bool any = false;
    for (int j = 0; j < count; ++j) {
        if (!on_pair[j]) continue;
        any = true;
        if (tasks[j].out_dtype != MXFP4_OUT_BF16 || (tasks[j].ldc * 2) % 16 != 0) return false;
    }
    if (!any || wide_clusters <= 0) return false;
    const int policy = g_tile_policy.load(std::memory_order_relaxed);
    if (policy != MXFP4_TILES_AUTO) return policy == MXFP4_TILES_WIDE;
    return pair_time_model(tasks, on_pair, count, wide_clusters, mxfp4::kPairTileNWide) <
           pair_time_model(tasks, on_pair, count, narrow_clusters, 256);
}

// ---- hybrid FP8 backward ------------------------------------------------------------

inline int64_t pad16(int64_t n) { return cdiv(n, 16) * 16; }
inline bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

mxfp4_status fp8_gemm_check(const mxfp4_fp8_gemm_task& t) {
    if (!t.a || !t.a_scale_inv || !t.b || !t.b_scale_inv || !t.c) return MXFP4_ERR_INVALID_ARG;
    if (t.M < 1 || t.N < 1 || t.K < 1 || t.M > kMaxDim || t.N > kMaxDim || t.K > kMaxDim)
        return MXFP4_ERR_INVALID_ARG;
    if (t.ldc < t.N || t.ldc > kMaxDim) return MXFP4_ERR_INVALID_ARG;
    if (t.out_dtype != MXFP4_OUT_BF16 && t.out_dtype != MXFP4_OUT_F32) return MXFP4_ERR_INVALID_ARG;
    if (!aligned16(t.a) || !aligned16(t.b) || !aligned16(t.c) || !aligned4(t.a_scale_inv) ||
        !aligned4(t.b_scale_inv))
        return MXFP4_ERR_MISALIGNED;
    return MXFP4_OK;
}

// Appends a checked FP8 GEMM to the batch: A / B maps over the codes (pitch round16(K)
// bytes, box 128 x 128, 128-byte swizzle) and C as for the MXFP4 GEMMs.
mxfp4_status fp8_gemm_fill(const mxfp4_fp8_gemm_task& t, DeviceState* dev, mxfp4::Fp8GemmBatch* b) {
    const int j = b->count;
    mxfp4::Fp8GemmArgs& g = b->args[j];
    const uint64_t ld = static_cast<uint64_t>(pad16(t.K));
    if (!encode_2d(&b->amap[j], CU_TENSOR_MAP_DATA_TYPE_UINT8, t.a, static_cast<uint64_t>(t.K),
                   static_cast<uint64_t>(t.M), ld, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&b->bmap[j], CU_TENSOR_MAP_DATA_TYPE_UINT8, t.b, static_cast<uint64_t>(t.K),
                   static_cast<uint64_t>(t.N), ld, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B))
        return MXFP4_ERR_CUDA;
    const int64_t esize = t.out_dtype == MXFP4_OUT_F32 ? 4 : 2;
    std::memset(&b->cmap[j], 0, sizeof(b->cmap[j]));
    const bool c_tma = (t.ldc * esize) % 16 == 0 &&
                       encode_2d(&b->cmap[j], t.out_dtype == MXFP4_OUT_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                                                          : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                                 t.c, static_cast<uint64_t>(t.N), static_cast<uint64_t>(t.M),
                                 static_cast<uint64_t>(t.ldc * esize), static_cast<uint32_t>(64 / esize), 32,
                                 CU_TENSOR_MAP_SWIZZLE_64B);
    g.M = t.M;
    g.N = t.N;
    g.tiles_m2 = static_cast<int32_t>(cdiv(t.M, 256));
    g.tiles_n = static_cast<int32_t>(cdiv(t.N, 256));
    g.k_stages = static_cast<int32_t>(cdiv(t.K, 128));
    g.c = t.c;
    g.ldc = t.ldc;
    g.out_f32 = t.out_dtype == MXFP4_OUT_F32 ? 1 : 0;
    g.c_tma = c_tma ? 1 : 0;
    g.a_scale_inv = t.a_scale_inv;
    g.b_scale_inv = t.b_scale_inv;
    g.err = dev->err;
    const int64_t before = j > 0 ? b->tile_end[j - 1] : 0;
    const int64_t end = before + static_cast<int64_t>(g.tiles_m2) * g.tiles_n;
    if (end > (int64_t{1} << 31) - 1) return MXFP4_ERR_INVALID_ARG;
    b->tile_end[j] = static_cast<int32_t>(end);
    b->count = j + 1;
    return MXFP4_OK;
}

}  // namespace

namespace mxfp4 {
cudaError_t launch_selftest_wait(uint32_t* err, uint64_t timeout_ns, cudaStream_t stream) {
    selftest_wait_kernel<<<1, 32, 0, stream>>>(err, timeout_ns);
    return cudaGetLastError();
}
}  // namespace mxfp4

extern "C" {

mxfp4_status mxfp4_quantize_sizes(int64_t rows, int64_t k, mxfp4_scale_layout layout, size_t* q_bytes,
                                  size_t* s_bytes) {
    if (rows < 1 || k < 1 || rows > kMaxDim || k > kMaxDim) return MXFP4_ERR_INVALID_ARG;
    if (layout != MXFP4_SCALE_PLAIN && layout != MXFP4_SCALE_TC) return MXFP4_ERR_INVALID_ARG;
    const int64_t kp = pad128(k);
    if (q_bytes) *q_bytes = static_cast<size_t>(rows) * static_cast<size_t>(kp / 2);
    if (s_bytes) {
        const int64_t r = layout == MXFP4_SCALE_TC ? pad128(rows) : rows;
        *s_bytes = static_cast<size_t>(r) * static_cast<size_t>(kp / 32);
    }
    return MXFP4_OK;
}

mxfp4_status mxfp4_quantize(const void* x, int64_t M, int64_t K, int64_t ldx, void* q_row, void* s_row,
                            mxfp4_scale_layout layout, mxfp4_stream_t stream) {
    return quantize_common(x, M, K, ldx, q_row, s_row, nullptr, nullptr, layout, false,
                           reinterpret_cast<cudaStream_t>(stream));
}

mxfp4_status mxfp4_quantize_dual(const void* x, int64_t M, int64_t K, int64_t ldx, void* q_row, void* s_row,
                                 void* q_col, void* s_col, mxfp4_scale_layout layout, mxfp4_stream_t stream) {
    return quantize_common(x, M, K, ldx, q_row, s_row, q_col, s_col, layout, true,
                           reinterpret_cast<cudaStream_t>(stream));
}

mxfp4_status mxfp4_quantize_dual_sr(const void* x, int64_t M, int64_t K, int64_t ldx, void* q_row, void* s_row,
                                    void* q_col, void* s_col, mxfp4_scale_layout layout, uint64_t seed,
                                    mxfp4_stream_t stream) {
    return quantize_common(x, M, K, ldx, q_row, s_row, q_col, s_col, layout, true,
                           reinterpret_cast<cudaStream_t>(stream), true, seed);
}

mxfp4_status mxfp4_quantize_dual_2d(const void* x, int64_t M, int64_t K, int64_t ldx, void* q_row, void* s_row,
                                    void* q_col, void* s_col, mxfp4_scale_layout layout, mxfp4_stream_t stream) {
    return quantize_common(x, M, K, ldx, q_row, s_row, q_col, s_col, layout, true,
                           reinterpret_cast<cudaStream_t>(stream), false, 0, MXFP4_QUANT_2D_BLOCKS);
}

mxfp4_status mxfp4_quantize_dual_rht(const void* x, int64_t M, int64_t K, int64_t ldx, void* q_row, void* s_row,
                                     void* q_col, void* s_col, mxfp4_scale_layout layout, uint32_t signs,
                                     mxfp4_stream_t stream) {
    return quantize_common(x, M, K, ldx, q_row, s_row, q_col, s_col, layout, true,
                           reinterpret_cast<cudaStream_t>(stream), false, 0, MXFP4_QUANT_RHT_COL, signs);
}

mxfp4_status mxfp4_quantize_dual_rht_sr(const void* x, int64_t M, int64_t K, int64_t ldx, void* q_row,
                                        void* s_row, void* q_col, void* s_col, mxfp4_scale_layout layout,
                                        uint32_t signs, uint64_t seed, mxfp4_stream_t stream) {
    return quantize_common(x, M, K, ldx, q_row, s_row, q_col, s_col, layout, true,
                           reinterpret_cast<cudaStream_t>(stream), true, seed, MXFP4_QUANT_RHT_COL, signs);
}

mxfp4_status mxfp4_quantize_dual_qk_norm_rope_bwd(const void* g, const void* x, int64_t M, int64_t H,
                                                  const float* rstd, const float* wq, const float* wk,
                                                  const float* cos_table, const float* sin_table, void* q_row,
                                                  void* s_row, void* q_col, void* s_col, mxfp4_scale_layout layout,
                                                  void* dmixed, mxfp4_stream_t stream) {
    if (H < 1 || H > kMaxDim / (3 * mxfp4::kNormRopeD)) return MXFP4_ERR_INVALID_ARG;
    const int64_t K = 3 * H * mxfp4::kNormRopeD;
    mxfp4_status st = quantize_check(g, M, K, K, q_row, s_row, q_col, s_col, layout, true);
    if (st != MXFP4_OK) return st;
    if (!x || !rstd || !wq || !wk || !cos_table || !sin_table) return MXFP4_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(cos_table) || !aligned16(sin_table) || (dmixed && !aligned16(dmixed)) ||
        (reinterpret_cast<uintptr_t>(rstd) & 3u) || (reinterpret_cast<uintptr_t>(wq) & 3u) ||
        (reinterpret_cast<uintptr_t>(wk) & 3u))
        return MXFP4_ERR_MISALIGNED;
    DeviceState* dev = nullptr;
    st = device_ready(&dev);
    if (st != MXFP4_OK) return st;
    mxfp4::QuantBatch b;
    std::memset(&b, 0, sizeof(b));
    st = quantize_task(g, M, K, K, q_row, s_row, q_col, s_col, layout, dev, &b, 0);
    if (st != MXFP4_OK) return st;
    mxfp4::NormRopeArgs a;
    std::memset(&a, 0, sizeof(a));
    a.gmap = b.maps[0];
    if (!encode_2d(&a.xmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, static_cast<uint64_t>(K), static_cast<uint64_t>(M),
                   static_cast<uint64_t>(K) * 2, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B))
        return MXFP4_ERR_CUDA;
    a.q = b.args[0];
    a.rstd = rstd;
    a.wq = wq;
    a.wk = wk;
    a.cosv = cos_table;
    a.sinv = sin_table;
    a.dmixed = static_cast<uint16_t*>(dmixed);
    a.H = static_cast<int32_t>(H);
    // Units of `span` consecutive tiles of one row block, about one unit per CTA.
    const int64_t tiles = static_cast<int64_t>(a.q.tiles_m) * a.q.tiles_k;
    const int64_t cap = static_cast<int64_t>(dev->sms) * mxfp4::quantize_norm_rope_ctas_per_sm();
    int64_t span = cdiv(tiles, cap) < a.q.tiles_k ? cdiv(tiles, cap) : a.q.tiles_k;
    if (span > 3 * mxfp4::kNormRopeMaxUnitHeads - 2) span = 3 * mxfp4::kNormRopeMaxUnitHeads - 2;
    a.span = static_cast<int32_t>(span);
    a.units_per_row = static_cast<int32_t>(cdiv(a.q.tiles_k, span));
    a.units = a.q.tiles_m * a.units_per_row;
    const int grid = static_cast<int>(a.units < cap ? a.units : cap);
    return mxfp4::launch_quantize_norm_rope(a, grid, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? MXFP4_OK
               : MXFP4_ERR_CUDA;
}

mxfp4_status mxfp4_quantize_batch(int32_t count, const mxfp4_quantize_task* tasks, int32_t dual,
                                  mxfp4_scale_layout layout, mxfp4_stream_t stream) {
    if (count < 1 || count > MXFP4_MAX_BATCH || tasks == nullptr) return MXFP4_ERR_INVALID_ARG;
    const bool d = dual != 0;
    for (int j = 0; j < count; ++j) {
        const mxfp4_quantize_task& t = tasks[j];
        const mxfp4_status st = quantize_check(t.x, t.rows, t.k, t.ldx, t.q_row, t.s_row, t.q_col, t.s_col,
                                               layout, d);
        if (st != MXFP4_OK) return st;
        if ((t.flags & ~(MXFP4_QUANT_2D_BLOCKS | MXFP4_QUANT_RHT_COL)) != 0 ||
            t.flags == (MXFP4_QUANT_2D_BLOCKS | MXFP4_QUANT_RHT_COL) || ((t.flags & MXFP4_QUANT_RHT_COL) && !d))
            return MXFP4_ERR_INVALID_ARG;
        if (t.amax != nullptr && d) return MXFP4_ERR_INVALID_ARG;   // row-only batches only
        if (t.amax != nullptr && (reinterpret_cast<uintptr_t>(t.amax) & 3u)) return MXFP4_ERR_MISALIGNED;
    }
    DeviceState* dev = nullptr;
    mxfp4_status st = device_ready(&dev);
    if (st != MXFP4_OK) return st;
    mxfp4::QuantBatch b;
    std::memset(&b, 0, sizeof(b));
    for (int j = 0; j < count; ++j) {
        const mxfp4_quantize_task& t = tasks[j];
        st = quantize_task(t.x, t.rows, t.k, t.ldx, t.q_row, t.s_row, t.q_col, t.s_col, layout, dev, &b, j,
                           t.flags, t.rht_signs);
        if (st != MXFP4_OK) return st;
        b.args[j].amax_bits = reinterpret_cast<uint32_t*>(t.amax);
    }
    return launch_batch(b, d, dev, reinterpret_cast<cudaStream_t>(stream));
}

mxfp4_status mxfp4_gemm(const void* a_q, const void* a_s, const void* b_q, const void* b_s, int64_t M, int64_t N,
                        int64_t K, void* c, int64_t ldc, mxfp4_out_dtype out_dtype, mxfp4_stream_t stream) {
    const mxfp4_gemm_task t{a_q, a_s, b_q, b_s, M, N, K, c, ldc, out_dtype, nullptr};
    return mxfp4_gemm_batch(1, &t, stream);
}

mxfp4_status mxfp4_gemm_bias(const void* a_q, const void* a_s, const void* b_q, const void* b_s, int64_t M,
                             int64_t N, int64_t K, const void* bias, void* c, int64_t ldc, mxfp4_out_dtype out_dtype,
                             mxfp4_stream_t stream) {
    if (bias == nullptr) return MXFP4_ERR_INVALID_ARG;
    const mxfp4_gemm_task t{a_q, a_s, b_q, b_s, M, N, K, c, ldc, out_dtype, bias};
    return mxfp4_gemm_batch(1, &t, stream);
}

mxfp4_status mxfp4_gemm_quantize(const void* a_q, const void* a_s, const void* b_q, const void* b_s, int64_t M,
                                 int64_t N, int64_t K, const void* bias, void* c, int64_t ldc, void* q_row, void* s_row,
                                 void* q_col, void* s_col, mxfp4_stream_t stream) {
    const mxfp4_gemm_task t{a_q, a_s, b_q, b_s, M, N, K, c, ldc, MXFP4_OUT_BF16, bias};
    mxfp4_status st = gemm_check(t);
    if (st != MXFP4_OK) return st;
    if (!q_row || !s_row || (q_col == nullptr) != (s_col == nullptr)) return MXFP4_ERR_INVALID_ARG;
    if ((ldc % 8) != 0 || !aligned16(q_row) || !aligned16(s_row) || (q_col && !aligned16(q_col)) ||
        (s_col && !aligned16(s_col)))
        return MXFP4_ERR_MISALIGNED;
    DeviceState* dev = nullptr;
    st = device_ready(&dev);
    if (st != MXFP4_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int max_clusters = mxfp4::gemm_pair_max_clusters(false);
    if (M <= mxfp4::kGemmBM || max_clusters <= 0) {
        // One 128-row tile: the one-CTA GEMM, then the quantizer over C (same bytes).
        st = mxfp4_gemm_batch(1, &t, stream);
        if (st != MXFP4_OK) return st;
        return quantize_common(c, M, N, ldc, q_row, s_row, q_col, s_col, MXFP4_SCALE_TC, q_col != nullptr, s);
    }
    mxfp4::GemmPairBatch b;
    std::memset(&b, 0, sizeof(b));
    st = gemm_fill_pair(t, dev, &b, false);
    if (st != MXFP4_OK) return st;
    mxfp4::GemmArgs& g = b.args[0];
    if (!g.c_tma) return MXFP4_ERR_CUDA;
    g.qo_row = static_cast<uint8_t*>(q_row);
    g.so_row = static_cast<uint8_t*>(s_row);
    g.qo_col = static_cast<uint8_t*>(q_col);
    g.so_col = static_cast<uint8_t*>(s_col);
    g.ldqo_row = pad128(N) / 2;
    g.ldqo_col = pad128(M) / 2;
    g.kb4o_row = static_cast<int32_t>(pad128(N) / 128);
    g.kb4o_col = static_cast<int32_t>(pad128(M) / 128);
    if (!encode_2d(&b.qrowmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, q_row, static_cast<uint64_t>(pad128(N) / 2),
                   static_cast<uint64_t>(M), static_cast<uint64_t>(pad128(N) / 2), 64, 32, CU_TENSOR_MAP_SWIZZLE_64B) ||
        (q_col != nullptr &&
         !encode_2d(&b.qcolmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, q_col, static_cast<uint64_t>(pad128(M) / 2),
                    static_cast<uint64_t>(N), static_cast<uint64_t>(pad128(M) / 2), 16, 128,
                    CU_TENSOR_MAP_SWIZZLE_NONE)))
        return MXFP4_ERR_CUDA;
    const int64_t tiles = b.tile_end[0];
    const int clusters = static_cast<int>(tiles < max_clusters ? tiles : max_clusters);
    return mxfp4::launch_gemm_pair(b, clusters, s, true, false) == cudaSuccess ? MXFP4_OK : MXFP4_ERR_CUDA;
}

mxfp4_status mxfp4_gemm_batch(int32_t count, const mxfp4_gemm_task* tasks, mxfp4_stream_t stream) {
    if (count < 1 || count > MXFP4_MAX_BATCH || tasks == nullptr) return MXFP4_ERR_INVALID_ARG;
    for (int j = 0; j < count; ++j) {
        const mxfp4_status st = gemm_check(tasks[j]);
        if (st != MXFP4_OK) return st;
    }
    DeviceState* dev = nullptr;
    mxfp4_status st = device_ready(&dev);
    if (st != MXFP4_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

    // Problems of more than one 128-row tile share one CTA-pair launch; the others run on
    // the one-CTA kernel, one launch each.  Every task's arguments and tensor maps are
    // prepared before the first launch, so a failing task leaves nothing enqueued.
    const int max_clusters = mxfp4::gemm_pair_max_clusters(false);
    bool on_pair[MXFP4_MAX_BATCH];
    for (int j = 0; j < count; ++j) on_pair[j] = tasks[j].M > mxfp4::kGemmBM && max_clusters > 0;
    const int wide_clusters = mxfp4::gemm_pair_max_clusters(true);
    const bool wide = pair_use_wide(tasks, on_pair, count, max_clusters, wide_clusters);
    mxfp4::GemmPairBatch b;
    std::memset(&b, 0, sizeof(b));
    struct Single {
        mxfp4::GemmArgs g;
        CUtensorMap amap, bmap, cmap;
    };
    Single singles[MXFP4_MAX_BATCH];
    int n_single = 0;
    for (int j = 0; j < count; ++j) {
        const mxfp4_gemm_task& t = tasks[j];
        if (on_pair[j]) {
            st = gemm_fill_pair(t, dev, &b, wide);
        } else {
            Single& o = singles[n_single++];
            st = gemm_fill(t, dev, &o.g, &o.amap, &o.bmap, &o.cmap, mxfp4::kGemmBN);
        }
        if (st != MXFP4_OK) return st;
    }
    for (int i = 0; i < n_single; ++i) {
        const Single& o = singles[i];
        const int64_t tiles = static_cast<int64_t>(o.g.tiles_m) * o.g.tiles_n;
        const int grid = static_cast<int>(tiles < dev->sms ? tiles : dev->sms);
        if (mxfp4::launch_gemm(o.amap, o.bmap, o.cmap, o.g, grid, s) != cudaSuccess) return MXFP4_ERR_CUDA;
    }
    if (b.count == 0) return MXFP4_OK;
    const int64_t pair_tiles = b.tile_end[b.count - 1];
    const int cmax = wide ? wide_clusters : max_clusters;
    const int clusters = static_cast<int>(pair_tiles < cmax ? pair_tiles : cmax);
    return mxfp4::launch_gemm_pair(b, clusters, s, false, wide) == cudaSuccess ? MXFP4_OK : MXFP4_ERR_CUDA;
}

mxfp4_status mxfp4_gemm_set_tile_policy(int32_t policy) {
    if (policy != MXFP4_TILES_AUTO && policy != MXFP4_TILES_NARROW && policy != MXFP4_TILES_WIDE)
        return MXFP4_ERR_INVALID_ARG;
    g_tile_policy.store(policy, std::memory_order_relaxed);
    return MXFP4_OK;
}

mxfp4_status mxfp4_fp8_quantize_tw_batch(int32_t count, const mxfp4_fp8_quantize_task* tasks,
                                         mxfp4_stream_t stream) {
    if (count < 1 || count > MXFP4_MAX_BATCH || tasks == nullptr) return MXFP4_ERR_INVALID_ARG;
    for (int j = 0; j < count; ++j) {
        const mxfp4_fp8_quantize_task& t = tasks[j];
        if (t.x == nullptr || (t.q_row == nullptr && t.q_col == nullptr) || t.amax == nullptr ||
            t.scale_inv == nullptr)
            return MXFP4_ERR_INVALID_ARG;
        if (t.M < 1 || t.K < 1 || t.M > kMaxDim || t.K > kMaxDim || t.ldx < t.K || t.ldx > kMaxDim)
            return MXFP4_ERR_INVALID_ARG;
        if (!aligned16(t.x) || (t.ldx % 8) != 0 || (t.q_row && !aligned16(t.q_row)) ||
            (t.q_col && !aligned16(t.q_col)) || !aligned4(t.amax) || !aligned4(t.scale_inv))
            return MXFP4_ERR_MISALIGNED;
    }
    DeviceState* dev = nullptr;
    const mxfp4_status st = device_ready(&dev);
    if (st != MXFP4_OK) return st;
    mxfp4::Fp8QuantBatch b;
    std::memset(&b, 0, sizeof(b));
    int64_t rows = 0, tiles = 0;
    for (int j = 0; j < count; ++j) {
        const mxfp4_fp8_quantize_task& t = tasks[j];
        b.t[j] = mxfp4::Fp8QuantArgs{t.x,        t.M,        t.K,    t.ldx,         t.q_row,
                                     pad16(t.K), t.q_col,    pad16(t.M), t.amax, t.scale_inv,
                                     t.amax_given != 0 ? 1 : 0};
        rows += t.M;
        tiles += cdiv(t.M, 64) * cdiv(t.K, 64);
        b.row_end[j] = rows;
        b.tile_end[j] = tiles;
    }
    b.count = count;
    b.err = dev->err;
    return mxfp4::launch_fp8_quantize(b, dev->sms, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? MXFP4_OK
               : MXFP4_ERR_CUDA;
}

mxfp4_status mxfp4_fp8_quantize_tw(const void* x, int64_t M, int64_t K, int64_t ldx, void* q_row, void* q_col,
                                   float* amax, float* scale_inv, mxfp4_stream_t stream) {
    const mxfp4_fp8_quantize_task t{x, M, K, ldx, q_row, q_col, amax, scale_inv};
    return mxfp4_fp8_quantize_tw_batch(1, &t, stream);
}

mxfp4_status mxfp4_fp8_gemm_batch(int32_t count, const mxfp4_fp8_gemm_task* tasks, mxfp4_stream_t stream) {
    if (count < 1 || count > MXFP4_MAX_BATCH || tasks == nullptr) return MXFP4_ERR_INVALID_ARG;
    for (int j = 0; j < count; ++j) {
        const mxfp4_status st = fp8_gemm_check(tasks[j]);
        if (st != MXFP4_OK) return st;
    }
    DeviceState* dev = nullptr;
    mxfp4_status st = device_ready(&dev);
    if (st != MXFP4_OK) return st;
    const int max_clusters = mxfp4::gemm_fp8_max_clusters();
    if (max_clusters < 1) return MXFP4_ERR_CUDA;
    mxfp4::Fp8GemmBatch b;
    std::memset(&b, 0, sizeof(b));
    for (int j = 0; j < count; ++j) {
        st = fp8_gemm_fill(tasks[j], dev, &b);
        if (st != MXFP4_OK) return st;
    }
    const int64_t tiles = b.tile_end[b.count - 1];
    const int clusters = static_cast<int>(tiles < max_clusters ? tiles : max_clusters);
    return mxfp4::launch_gemm_fp8(b, clusters, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? MXFP4_OK
               : MXFP4_ERR_CUDA;
}

mxfp4_status mxfp4_fp8_gemm(const void* a, const float* a_scale_inv, const void* b, const float* b_scale_inv,
                            int64_t M, int64_t N, int64_t K, void* c, int64_t ldc, mxfp4_out_dtype out_dtype,
                            mxfp4_stream_t stream) {
    const mxfp4_fp8_gemm_task t{a, a_scale_inv, b, b_scale_inv, M, N, K, c, ldc, out_dtype};
    return mxfp4_fp8_gemm_batch(1, &t, stream);
}

mxfp4_status mxfp4_last_device_error(mxfp4_stream_t stream) {
    DeviceState* dev = nullptr;
    mxfp4_status st = device_ready(&dev);
    if (st != MXFP4_OK) return st;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return MXFP4_ERR_CUDA;
    uint32_t word = 0;
    if (cudaMemcpy(&word, dev->err, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return MXFP4_ERR_CUDA;
    if (word != 0) {
        const uint32_t zero = 0;
        if (cudaMemcpy(dev->err, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return MXFP4_ERR_CUDA;
        return (word & mxfp4::kErrWaitBits) ? MXFP4_ERR_TIMEOUT : MXFP4_ERR_NONFINITE;
    }
    return MXFP4_OK;
}

mxfp4_status mxfp4_selftest_bounded_wait(int64_t timeout_ns, mxfp4_stream_t stream) {
    if (timeout_ns < 1 || timeout_ns > 10000000000LL) return MXFP4_ERR_INVALID_ARG;
    DeviceState* dev = nullptr;
    mxfp4_status st = device_ready(&dev);
    if (st != MXFP4_OK) return st;
    return mxfp4::launch_selftest_wait(dev->err, static_cast<uint64_t>(timeout_ns),
                                       reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? MXFP4_OK
               : MXFP4_ERR_CUDA;
}

const char* mxfp4_status_string(mxfp4_status status) {
    switch (status) {
        case MXFP4_OK: return "MXFP4_OK";
        case MXFP4_ERR_INVALID_ARG: return "MXFP4_ERR_INVALID_ARG: a size, pitch, pointer or enum is out of range";
        case MXFP4_ERR_MISALIGNED: return "MXFP4_ERR_MISALIGNED: a pointer or pitch breaks the 16-byte rule";
        case MXFP4_ERR_UNSUPPORTED_DEVICE:
            return "MXFP4_ERR_UNSUPPORTED_DEVICE: the current device is not compute capability 10.3 (sm_103)";
        case MXFP4_ERR_CUDA: return "MXFP4_ERR_CUDA: a CUDA call or kernel launch failed";
        case MXFP4_ERR_TIMEOUT: return "MXFP4_ERR_TIMEOUT: a kernel's bounded wait ran out";
        case MXFP4_ERR_NONFINITE:
            return "MXFP4_ERR_NONFINITE: a tensorwise FP8 quantization met a NaN or infinite input";
    }
    return "MXFP4: unknown status";
}

}  // extern "C"
