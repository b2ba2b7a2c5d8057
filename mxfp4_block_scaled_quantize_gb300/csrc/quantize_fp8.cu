// quantize_fp8.cu -- tensorwise FP8 (E5M2) quantization for the hybrid backward.
//
// `MXFP4LinearFunction.backward` in primus_turbo_mxfp4_local.py, with `backward_is_fp8`,
// quantizes dY, X and W with `_quantize_fp8_tw(…, float8_e5m2)` (one scale per tensor)
// and runs dgrad / wgrad as FP8 GEMMs.  The pages do not define `_quantize_fp8_tw`; this
// follows the usual tensorwise recipe: amax = max |x|; scale = 57344 / amax in fp32 (the
// largest finite fp32 if that overflows, 1 for amax = 0); element = E5M2 round-to-nearest-
// even of x * scale (fp32 product), saturating at +-57344; scale_inv = 1 / scale.
//
// Up to four tensors per call: the amax words are zeroed, then for each tensor an amax
// pass (each warp folds its maxima into the tensor's amax word with one atomicMax on the
// fp32 bit pattern, which orders like the value for non-negative floats; skipped, and the
// word left alone, for a tensor whose amax an earlier MXFP4 quantization wrote) and a conversion
// pass over 64 x 64 tiles that writes the row copy (X's codes, row pitch
// ldr bytes) and/or the column copy (X^T's codes, row pitch ldc bytes) through a shared
// transpose, so both copies leave in 16-byte row pieces.  The column copies are what keep
// the FP8 GEMMs in the same K-major ("TN") form as the MXFP4 ones: dgrad reads W^T, wgrad
// dY^T and X^T.
#include <cfloat>
#include <cuda_bf16.h>
#include <cstdint>

#include "launch_fp8.h"
#include "ptx.cuh"

namespace mxfp4 {
namespace {

constexpr int kFt = 64;            // tile edge
constexpr int kFThreads = 256;     // 4 threads per tile row, 16 elements each

__global__ void fp8_zero_kernel(const __grid_constant__ Fp8QuantBatch B) {
    if (static_cast<int>(threadIdx.x) < B.count && !B.t[threadIdx.x].amax_given) *B.t[threadIdx.x].amax = 0.0f;
}

// 16 bytes through the read-only path with an L2 eviction-priority policy.
__device__ __forceinline__ uint4 ldg16_policy(const void* p, uint64_t pol) {
    uint4 v;
    asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p), "l"(pol));
    return v;
}

// One warp per row at a time (rows of all tasks in sequence, task of a row by row_end),
// its lanes across the row's 8-element chunks, four independent 16-byte loads in flight
// per lane; no division on the hot path.
__global__ void __launch_bounds__(256) fp8_amax_kernel(const __grid_constant__ Fp8QuantBatch B) {
    uint32_t m[kMaxFp8Tasks] = {0u, 0u, 0u, 0u};   // per task: largest |x| as bf16 magnitude bits
    // The conversion pass reads the tensor again right after this one: keep it in L2.
    const uint64_t pol = l2_policy_evict_last();
    const int64_t rows = B.row_end[B.count - 1];
    const int lane = threadIdx.x & 31;
    const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    int j = 0;
    for (int64_t g = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; g < rows; g += warps) {
        while (j + 1 < B.count && g >= B.row_end[j]) ++j;   // rows only grow along the loop
        const Fp8QuantArgs& a = B.t[j];
        const int64_t r = g - (j > 0 ? B.row_end[j - 1] : 0);
        const uint16_t* const row = static_cast<const uint16_t*>(a.x) + r * a.ldx;
        const int64_t K = a.K;
        uint32_t v = 0;
        for (int64_t c0 = static_cast<int64_t>(lane) * 8; c0 < K; c0 += 32 * 8 * 4) {
            uint4 q[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int64_t c = c0 + u * 32 * 8;
                q[u] = c + 8 <= K ? ldg16_policy(row + c, pol) : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint32_t w[4] = {q[u].x, q[u].y, q[u].z, q[u].w};
#pragma unroll
                for (int k = 0; k < 4; ++k) v = max(v, max(w[k] & 0x7FFFu, (w[k] >> 16) & 0x7FFFu));
                const int64_t c = c0 + u * 32 * 8;
                if (c < K && c + 8 > K)   // the row's ragged last chunk
                    for (int64_t k = 0; c + k < K; ++k) v = max(v, static_cast<uint32_t>(__ldg(row + c + k)) & 0x7FFFu);
            }
        }
#pragma unroll
        for (int k = 0; k < kMaxFp8Tasks; ++k)
            if (k == j) m[k] = max(m[k], v);
    }
#pragma unroll
    for (int k = 0; k < kMaxFp8Tasks; ++k) {
        if (k >= B.count) break;
        const uint32_t w = __reduce_max_sync(0xFFFFFFFFu, m[k]);
        if (lane == 0 && w != 0) atomicMax(reinterpret_cast<uint32_t*>(B.t[k].amax), w << 16);
    }
}

__device__ __forceinline__ uint32_t e5m2x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ float tensor_scale(float amax) {
    float scale = 1.0f;
    if (amax > 0.0f) {
        scale = __fdiv_rn(57344.0f, amax);
        if (isinf(scale)) scale = FLT_MAX;
    }
    return scale;
}

// Task and first row / column of launch tile tg (row-major 64 x 64 tiles of each task);
// one 32-bit division per tile.
__device__ __forceinline__ void tile_ref(const Fp8QuantBatch& B, int64_t tg, int* j, int64_t* m0, int64_t* k0) {
    int jj = 0;
    while (jj + 1 < B.count && tg >= B.tile_end[jj]) ++jj;
    const uint32_t tl = static_cast<uint32_t>(tg - (jj > 0 ? B.tile_end[jj - 1] : 0));
    const uint32_t tiles_k = static_cast<uint32_t>((B.t[jj].K + kFt - 1) / kFt);
    const uint32_t mt = tl / tiles_k;
    *j = jj;
    *m0 = static_cast<int64_t>(mt) * kFt;
    *k0 = static_cast<int64_t>(tl - mt * tiles_k) * kFt;
}

// The 16 elements that thread (r, c) converts in the tile at (m0, k0) of task j: row
// m0 + r, columns k0 + c .. + 15 (zero outside the tensor).
__device__ __forceinline__ void load_piece(const Fp8QuantBatch& B, int j, int64_t m0, int64_t k0, int r, int c,
                                           uint32_t* w) {
    const Fp8QuantArgs& a = B.t[j];
    const int64_t row = m0 + r, col = k0 + c;
    const uint16_t* p = static_cast<const uint16_t*>(a.x) + row * a.ldx + col;
    if (row < a.M && col + 16 <= a.K) {
        const uint64_t pol = l2_policy_evict_first();   // the tensor's last read
        const uint4 va = ldg16_policy(p, pol);
        const uint4 vb = ldg16_policy(p + 8, pol);
        w[0] = va.x; w[1] = va.y; w[2] = va.z; w[3] = va.w;
        w[4] = vb.x; w[5] = vb.y; w[6] = vb.z; w[7] = vb.w;
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const uint32_t lo = (row < a.M && col + 2 * e < a.K) ? __ldg(p + 2 * e) : 0u;
            const uint32_t hi = (row < a.M && col + 2 * e + 1 < a.K) ? __ldg(p + 2 * e + 1) : 0u;
            w[e] = lo | (hi << 16);
        }
    }
}

__global__ void __launch_bounds__(kFThreads) fp8_quantize_kernel(const __grid_constant__ Fp8QuantBatch B) {
    // 16-byte chunk j of tile row r sits at chunk j ^ ((r / 16) % 4): the column reads below
    // take one byte from rows 16 apart in each quarter of the warp, which then fall in four
    // different bank groups.
    __shared__ __align__(16) uint8_t tile[kFt][kFt];
    if (blockIdx.x == 0 && static_cast<int>(threadIdx.x) < B.count) {
        const Fp8QuantArgs& a = B.t[threadIdx.x];
        // amax is the fp32 pattern of a bf16 magnitude: NaN and inf sit at and above 0x7F800000
        if (*reinterpret_cast<const uint32_t*>(a.amax) >= 0x7F800000u) atomicOr(B.err, kErrNonFinite);
        *a.scale_inv = __fdiv_rn(1.0f, tensor_scale(*a.amax));
    }
    const int t = threadIdx.x;
    const int r = t >> 2, c = (t & 3) * 16;
    const int64_t tiles = B.tile_end[B.count - 1];
    // Tiles are taken from the end of the tensor backwards: the amax pass has just read the
    // tensor front to back (keeping it in L2 with priority), so its end is surely still there.
    float scales[kMaxFp8Tasks];
#pragma unroll
    for (int k = 0; k < kMaxFp8Tasks; ++k) scales[k] = k < B.count ? tensor_scale(*B.t[k].amax) : 1.0f;
    uint32_t next[8];
    int nj = 0;
    int64_t nm0 = 0, nk0 = 0;
    if (static_cast<int64_t>(blockIdx.x) < tiles) {
        tile_ref(B, tiles - 1 - blockIdx.x, &nj, &nm0, &nk0);
        load_piece(B, nj, nm0, nk0, r, c, next);
    }
    for (int64_t i = blockIdx.x; i < tiles; i += gridDim.x) {
        const int j = nj;
        const int64_t m0 = nm0, k0 = nk0;
        uint32_t w[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) w[e] = next[e];
        // the next tile's loads go out before this tile's stores and barriers
        if (i + gridDim.x < tiles) {
            tile_ref(B, tiles - 1 - (i + gridDim.x), &nj, &nm0, &nk0);
            load_piece(B, nj, nm0, nk0, r, c, next);
        }
        const Fp8QuantArgs& a = B.t[j];
        const int64_t M = a.M, K = a.K, ldr = a.ldr, ldc = a.ldc;
        uint8_t* const q_row = static_cast<uint8_t*>(a.q_row);
        uint8_t* const q_col = static_cast<uint8_t*>(a.q_col);
        float scale = scales[0];
#pragma unroll
        for (int k = 1; k < kMaxFp8Tasks; ++k)
            if (k == j) scale = scales[k];
        const int64_t row = m0 + r, col = k0 + c;
        uint32_t q[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const uint32_t e01 = e5m2x2(__fmul_rn(__uint_as_float(w[2 * e] << 16), scale),
                                        __fmul_rn(__uint_as_float(w[2 * e] & 0xFFFF0000u), scale));
            const uint32_t e23 = e5m2x2(__fmul_rn(__uint_as_float(w[2 * e + 1] << 16), scale),
                                        __fmul_rn(__uint_as_float(w[2 * e + 1] & 0xFFFF0000u), scale));
            q[e] = e01 | (e23 << 16);
        }
        if (q_row != nullptr && row < M && col < ldr)
            *reinterpret_cast<uint4*>(q_row + row * ldr + col) = make_uint4(q[0], q[1], q[2], q[3]);
        if (q_col != nullptr) {
            *reinterpret_cast<uint4*>(&tile[r][(((c >> 4) ^ ((r >> 4) & 3)) << 4)]) = make_uint4(q[0], q[1], q[2], q[3]);
            __syncthreads();
            // thread t: column k0 + (t >> 2), rows m0 + c .. + 15 of the tile (all in row
            // group c / 16, so one swizzled byte offset serves the 16 reads)
            const int kc = t >> 2;
            const int kb = (((kc >> 4) ^ (c >> 4)) << 4) | (kc & 15);
            uint32_t o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
                o[e] = static_cast<uint32_t>(tile[c + 4 * e][kb]) | (static_cast<uint32_t>(tile[c + 4 * e + 1][kb]) << 8) |
                       (static_cast<uint32_t>(tile[c + 4 * e + 2][kb]) << 16) |
                       (static_cast<uint32_t>(tile[c + 4 * e + 3][kb]) << 24);
            const int64_t krow = k0 + kc, mcol = m0 + c;
            if (krow < K && mcol < ldc)
                *reinterpret_cast<uint4*>(q_col + krow * ldc + mcol) = make_uint4(o[0], o[1], o[2], o[3]);
            __syncthreads();   // the tile is rewritten by the next iteration
        }
    }
}

}  // namespace

cudaError_t launch_fp8_quantize(const Fp8QuantBatch& b, int sms, cudaStream_t stream) {
    bool any_amax = false;
    for (int j = 0; j < b.count; ++j) any_amax = any_amax || !b.t[j].amax_given;
    cudaError_t e;
    if (any_amax) {
        fp8_zero_kernel<<<1, 32, 0, stream>>>(b);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    auto convert = [&](const Fp8QuantBatch& sub) {
        const int64_t tiles = sub.tile_end[sub.count - 1];
        const int grid2 = static_cast<int>(tiles < int64_t{sms} * 8 ? tiles : int64_t{sms} * 8);
        fp8_quantize_kernel<<<grid2, kFThreads, 0, stream>>>(sub);
        return cudaGetLastError();
    };
    // A tensor whose amax is still to be found: its amax pass, then its conversion pass right
    // away, which re-reads the tensor the amax pass has just streamed through L2 instead of
    // one the amax pass over all tensors has long evicted.
    Fp8QuantBatch given = b;
    given.count = 0;
    for (int j = 0; j < b.count; ++j) {
        const int64_t rows = b.row_end[j] - (j > 0 ? b.row_end[j - 1] : 0);
        const int64_t tiles = b.tile_end[j] - (j > 0 ? b.tile_end[j - 1] : 0);
        if (b.t[j].amax_given) {
            // the tensors whose amax is known convert together, in one launch, last
            const int k = given.count++;
            given.t[k] = b.t[j];
            given.row_end[k] = (k > 0 ? given.row_end[k - 1] : 0) + rows;
            given.tile_end[k] = (k > 0 ? given.tile_end[k - 1] : 0) + tiles;
            continue;
        }
        Fp8QuantBatch one = b;
        one.count = 1;
        one.t[0] = b.t[j];
        one.row_end[0] = rows;
        one.tile_end[0] = tiles;
        const int64_t want = (rows + 7) / 8;   // 8 warps per CTA, one row each
        const int grid1 = static_cast<int>(want < int64_t{sms} * 8 ? want : int64_t{sms} * 8);
        fp8_amax_kernel<<<grid1 > 0 ? grid1 : 1, 256, 0, stream>>>(one);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        e = convert(one);
        if (e != cudaSuccess) return e;
    }
    if (given.count > 0) {
        e = convert(given);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace mxfp4
