// api.cu -- the C ABI declared in include/mxfp4.h: argument checks, the device gate, TMA
// descriptor set-up and kernel launches.  Nothing here allocates device memory or
// synchronizes, except mxfp4_last_device_error, whose job is to synchronize.
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "launch.h"
#include "mxfp4.h"
#include "ptx.cuh"

namespace {

// Device error word: kernels OR a site bit into it when a bounded wait runs out.
__device__ uint32_t g_error_word;

constexpr int kMaxDevices = 64;
constexpr int64_t kMaxDim = (int64_t{1} << 31) - 512;  // keeps tile coordinates in int32

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
                           mxfp4::QuantBatch* b, int j) {
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
    a.err = dev->err;
    const int64_t before = j > 0 ? b->tile_end[j - 1] : 0;
    const int64_t end = before + static_cast<int64_t>(a.tiles_m) * a.tiles_k;
    if (end > (int64_t{1} << 31) - 1) return MXFP4_ERR_INVALID_ARG;
    b->tile_end[j] = static_cast<int32_t>(end);
    b->count = j + 1;
    return MXFP4_OK;
}

mxfp4_status launch_batch(const mxfp4::QuantBatch& b, bool dual, DeviceState* dev, cudaStream_t stream) {
    const int64_t tiles = b.tile_end[b.count - 1];
    const int64_t cap = static_cast<int64_t>(dev->sms) * mxfp4::quantize_ctas_per_sm();
    const int grid = static_cast<int>(tiles < cap ? tiles : cap);
    return mxfp4::launch_quantize(b, dual, grid, stream) == cudaSuccess ? MXFP4_OK : MXFP4_ERR_CUDA;
}

mxfp4_status quantize_common(const void* x, int64_t M, int64_t K, int64_t ldx, void* q_row, void* s_row,
                             void* q_col, void* s_col, mxfp4_scale_layout layout, bool dual,
                             cudaStream_t stream) {
    mxfp4_status st = quantize_check(x, M, K, ldx, q_row, s_row, q_col, s_col, layout, dual);
    if (st != MXFP4_OK) return st;
    DeviceState* dev = nullptr;
    st = device_ready(&dev);
    if (st != MXFP4_OK) return st;
    mxfp4::QuantBatch b;
    std::memset(&b, 0, sizeof(b));
    st = quantize_task(x, M, K, ldx, q_row, s_row, q_col, s_col, layout, dev, &b, 0);
    if (st != MXFP4_OK) return st;
    return launch_batch(b, dual, dev, stream);
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

mxfp4_status mxfp4_quantize_batch(int32_t count, const mxfp4_quantize_task* tasks, int32_t dual,
                                  mxfp4_scale_layout layout, mxfp4_stream_t stream) {
    if (count < 1 || count > MXFP4_MAX_BATCH || tasks == nullptr) return MXFP4_ERR_INVALID_ARG;
    const bool d = dual != 0;
    for (int j = 0; j < count; ++j) {
        const mxfp4_quantize_task& t = tasks[j];
        const mxfp4_status st = quantize_check(t.x, t.rows, t.k, t.ldx, t.q_row, t.s_row, t.q_col, t.s_col,
                                               layout, d);
        if (st != MXFP4_OK) return st;
    }
    DeviceState* dev = nullptr;
    mxfp4_status st = device_ready(&dev);
    if (st != MXFP4_OK) return st;
    mxfp4::QuantBatch b;
    std::memset(&b, 0, sizeof(b));
    for (int j = 0; j < count; ++j) {
        const mxfp4_quantize_task& t = tasks[j];
        st = quantize_task(t.x, t.rows, t.k, t.ldx, t.q_row, t.s_row, t.q_col, t.s_col, layout, dev, &b, j);
        if (st != MXFP4_OK) return st;
    }
    return launch_batch(b, d, dev, reinterpret_cast<cudaStream_t>(stream));
}

mxfp4_status mxfp4_gemm(const void* a_q, const void* a_s, const void* b_q, const void* b_s, int64_t M, int64_t N,
                        int64_t K, void* c, int64_t ldc, mxfp4_out_dtype out_dtype, mxfp4_stream_t stream) {
    if (!a_q || !a_s || !b_q || !b_s || !c) return MXFP4_ERR_INVALID_ARG;
    if (M < 1 || N < 1 || K < 1 || M > kMaxDim || N > kMaxDim || K > kMaxDim) return MXFP4_ERR_INVALID_ARG;
    if (ldc < N || ldc > kMaxDim) return MXFP4_ERR_INVALID_ARG;
    if (out_dtype != MXFP4_OUT_BF16 && out_dtype != MXFP4_OUT_F32) return MXFP4_ERR_INVALID_ARG;
    if (!aligned16(a_q) || !aligned16(a_s) || !aligned16(b_q) || !aligned16(b_s) || !aligned16(c))
        return MXFP4_ERR_MISALIGNED;
    DeviceState* dev = nullptr;
    mxfp4_status st = device_ready(&dev);
    if (st != MXFP4_OK) return st;

    const int64_t kp = pad128(K);
    CUtensorMap amap, bmap;
    if (!encode_2d(&amap, CU_TENSOR_MAP_DATA_TYPE_UINT8, a_q, static_cast<uint64_t>(kp / 2), static_cast<uint64_t>(M),
                   static_cast<uint64_t>(kp / 2), 128, mxfp4::kGemmBM, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&bmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, b_q, static_cast<uint64_t>(kp / 2), static_cast<uint64_t>(N),
                   static_cast<uint64_t>(kp / 2), 128, mxfp4::kGemmBN, CU_TENSOR_MAP_SWIZZLE_128B))
        return MXFP4_ERR_CUDA;

    // C goes out through TMA stores when its base and pitch allow a tensor map (16-byte
    // aligned base, pitch a multiple of 16 bytes); otherwise with plain stores.
    const int64_t esize = out_dtype == MXFP4_OUT_F32 ? 4 : 2;
    CUtensorMap cmap;
    std::memset(&cmap, 0, sizeof(cmap));
    const bool c_tma = (ldc * esize) % 16 == 0 &&
                       encode_2d(&cmap, out_dtype == MXFP4_OUT_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                                                   : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                                 c, static_cast<uint64_t>(N), static_cast<uint64_t>(M),
                                 static_cast<uint64_t>(ldc * esize), static_cast<uint32_t>(64 / esize), 32,
                                 CU_TENSOR_MAP_SWIZZLE_64B);

    mxfp4::GemmArgs g;
    g.M = M;
    g.N = N;
    g.tiles_m = static_cast<int32_t>(cdiv(M, mxfp4::kGemmBM));
    g.tiles_n = static_cast<int32_t>(cdiv(N, mxfp4::kGemmBN));
    g.k_stages = static_cast<int32_t>(cdiv(kp, 256));
    g.kb4 = static_cast<int32_t>(kp / 128);
    g.groups_b = static_cast<int32_t>(cdiv(N, 128));
    g.a_s = static_cast<const uint8_t*>(a_s);
    g.b_s = static_cast<const uint8_t*>(b_s);
    g.c = c;
    g.ldc = ldc;
    g.out_f32 = out_dtype == MXFP4_OUT_F32 ? 1 : 0;
    g.c_tma = c_tma ? 1 : 0;
    g.err = dev->err;
    g.tiles_m2 = static_cast<int32_t>(cdiv(M, 256));
    const int64_t tiles = static_cast<int64_t>(g.tiles_m) * g.tiles_n;
    if (tiles > (int64_t{1} << 31) - 1) return MXFP4_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

    // More than one 128-row tile: 256 x 256 tiles on CTA pairs.
    const int max_clusters = M > mxfp4::kGemmBM ? mxfp4::gemm_pair_max_clusters() : 0;
    if (max_clusters > 0) {
        CUtensorMap bmap2, sfamap, sfbmap;
        if (!encode_2d(&bmap2, CU_TENSOR_MAP_DATA_TYPE_UINT8, b_q, static_cast<uint64_t>(kp / 2),
                       static_cast<uint64_t>(N), static_cast<uint64_t>(kp / 2), 128, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_2d(&sfamap, CU_TENSOR_MAP_DATA_TYPE_UINT64, a_s, static_cast<uint64_t>(g.kb4) * 64,
                       static_cast<uint64_t>(cdiv(M, 128)), static_cast<uint64_t>(g.kb4) * 512, 128, 1,
                       CU_TENSOR_MAP_SWIZZLE_NONE) ||
            !encode_2d(&sfbmap, CU_TENSOR_MAP_DATA_TYPE_UINT64, b_s, static_cast<uint64_t>(g.kb4) * 64,
                       static_cast<uint64_t>(cdiv(N, 128)), static_cast<uint64_t>(g.kb4) * 512, 128, 2,
                       CU_TENSOR_MAP_SWIZZLE_NONE))
            return MXFP4_ERR_CUDA;
        const int64_t pair_tiles = static_cast<int64_t>(g.tiles_m2) * g.tiles_n;
        const int clusters = static_cast<int>(pair_tiles < max_clusters ? pair_tiles : max_clusters);
        return mxfp4::launch_gemm_pair(amap, bmap2, cmap, sfamap, sfbmap, g, clusters, s) == cudaSuccess
                   ? MXFP4_OK
                   : MXFP4_ERR_CUDA;
    }
    const int grid = static_cast<int>(tiles < dev->sms ? tiles : dev->sms);
    return mxfp4::launch_gemm(amap, bmap, cmap, g, grid, s) == cudaSuccess ? MXFP4_OK : MXFP4_ERR_CUDA;
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
        return MXFP4_ERR_TIMEOUT;
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
    }
    return "MXFP4: unknown status";
}

}  // extern "C"
