// quantize_fp8.cu -- tensorwise FP8 (E5M2) quantization for the hybrid backward.
//
// `MXFP4LinearFunction.backward` in primus_turbo_mxfp4_local.py, with `backward_is_fp8`,
// quantizes dY, X and W with `_quantize_fp8_tw(…, float8_e5m2)` (one scale per tensor)
// and runs dgrad / wgrad as FP8 GEMMs.  The pages do not define `_quantize_fp8_tw`; this
// follows the usual tensorwise recipe: amax = max |x|; scale = 57344 / amax in fp32 (the
// largest finite fp32 if that overflows, 1 for amax = 0); element = E5M2 round-to-nearest-
// even of x * scale (fp32 product), saturating at +-57344; scale_inv = 1 / scale.
//
// Two launches: an amax pass (each warp folds its maximum into the output amax with one
// atomicMax on the fp32 bit pattern, which orders like the value for non-negative floats)
// and a conversion pass over 64 x 64 tiles that writes the row copy (X's codes, row pitch
// ldr bytes) and/or the column copy (X^T's codes, row pitch ldc bytes) through a shared
// transpose, so both copies leave in 16-byte row pieces.  The column copies are what keep
// the FP8 GEMMs in the same K-major ("TN") form as the MXFP4 ones: dgrad reads W^T, wgrad
// dY^T and X^T.
#include <cfloat>
#include <cuda_bf16.h>
#include <cstdint>

#include "launch_fp8.h"

namespace mxfp4 {
namespace {

constexpr int kFt = 64;            // tile edge
constexpr int kFThreads = 256;     // 4 threads per tile row, 16 elements each

__global__ void __launch_bounds__(256) fp8_amax_kernel(const uint16_t* __restrict__ x, int64_t M, int64_t K,
                                                        int64_t ldx, uint32_t* amax_bits) {
    uint32_t m = 0;   // largest |x| as fp32 bits (bf16 magnitude bits << 16)
    const int64_t chunks = (K + 7) / 8;
    const int64_t total = M * chunks;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = i / chunks, c = (i % chunks) * 8;
        const uint16_t* p = x + r * ldx + c;
        if (c + 8 <= K) {
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) m = max(m, max(w[j] & 0x7FFFu, (w[j] >> 16) & 0x7FFFu));
        } else {
            for (int64_t j = 0; c + j < K; ++j) m = max(m, static_cast<uint32_t>(__ldg(p + j)) & 0x7FFFu);
        }
    }
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    if ((threadIdx.x & 31) == 0 && m != 0) atomicMax(amax_bits, m << 16);
}

__device__ __forceinline__ uint32_t e5m2x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

__global__ void __launch_bounds__(kFThreads) fp8_quantize_kernel(const uint16_t* __restrict__ x, int64_t M, int64_t K,
                                                                 int64_t ldx, uint8_t* q_row, int64_t ldr,
                                                                 uint8_t* q_col, int64_t ldc, const float* amax_p,
                                                                 float* scale_inv_p) {
    __shared__ __align__(16) uint8_t tile[kFt][kFt + 16];
    const float amax = *amax_p;
    float scale = 1.0f;
    if (amax > 0.0f) {
        scale = __fdiv_rn(57344.0f, amax);
        if (isinf(scale)) scale = FLT_MAX;
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) *scale_inv_p = __fdiv_rn(1.0f, scale);

    const int t = threadIdx.x;
    const int r = t >> 2, c = (t & 3) * 16;
    const int64_t tiles_k = (K + kFt - 1) / kFt;
    const int64_t tiles = ((M + kFt - 1) / kFt) * tiles_k;
    for (int64_t tl = blockIdx.x; tl < tiles; tl += gridDim.x) {
        const int64_t m0 = (tl / tiles_k) * kFt, k0 = (tl % tiles_k) * kFt;
        // 16 elements of row m0 + r, columns k0 + c .. + 15 (zero outside X)
        uint32_t w[8];
        const int64_t row = m0 + r, col = k0 + c;
        const uint16_t* p = x + row * ldx + col;
        if (row < M && col + 16 <= K) {
            const uint4 a = __ldg(reinterpret_cast<const uint4*>(p));
            const uint4 b = __ldg(reinterpret_cast<const uint4*>(p + 8));
            w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
            w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const uint32_t lo = (row < M && col + 2 * j < K) ? __ldg(p + 2 * j) : 0u;
                const uint32_t hi = (row < M && col + 2 * j + 1 < K) ? __ldg(p + 2 * j + 1) : 0u;
                w[j] = lo | (hi << 16);
            }
        }
        uint32_t q[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t e01 = e5m2x2(__fmul_rn(__uint_as_float(w[2 * j] << 16), scale),
                                        __fmul_rn(__uint_as_float(w[2 * j] & 0xFFFF0000u), scale));
            const uint32_t e23 = e5m2x2(__fmul_rn(__uint_as_float(w[2 * j + 1] << 16), scale),
                                        __fmul_rn(__uint_as_float(w[2 * j + 1] & 0xFFFF0000u), scale));
            q[j] = e01 | (e23 << 16);
        }
        if (q_row != nullptr && row < M && col < ldr)
            *reinterpret_cast<uint4*>(q_row + row * ldr + col) = make_uint4(q[0], q[1], q[2], q[3]);
        if (q_col != nullptr) {
            *reinterpret_cast<uint4*>(&tile[r][c]) = make_uint4(q[0], q[1], q[2], q[3]);
            __syncthreads();
            // thread t: column k0 + (t >> 2), rows m0 + c .. + 15 of the tile
            const int kc = t >> 2;
            uint32_t o[4];
#pragma unroll
            for (int j = 0; j < 4; ++j)
                o[j] = static_cast<uint32_t>(tile[c + 4 * j][kc]) | (static_cast<uint32_t>(tile[c + 4 * j + 1][kc]) << 8) |
                       (static_cast<uint32_t>(tile[c + 4 * j + 2][kc]) << 16) |
                       (static_cast<uint32_t>(tile[c + 4 * j + 3][kc]) << 24);
            const int64_t krow = k0 + kc, mcol = m0 + c;
            if (krow < K && mcol < ldc)
                *reinterpret_cast<uint4*>(q_col + krow * ldc + mcol) = make_uint4(o[0], o[1], o[2], o[3]);
            __syncthreads();   // the tile is rewritten by the next iteration
        }
    }
}

}  // namespace

cudaError_t launch_fp8_quantize(const Fp8QuantArgs& a, int sms, cudaStream_t stream) {
    cudaError_t e = cudaMemsetAsync(a.amax, 0, sizeof(float), stream);
    if (e != cudaSuccess) return e;
    const int64_t chunks = a.M * ((a.K + 7) / 8);
    const int64_t want = (chunks + 255) / 256;
    const int grid1 = static_cast<int>(want < int64_t{sms} * 8 ? want : int64_t{sms} * 8);
    fp8_amax_kernel<<<grid1 > 0 ? grid1 : 1, 256, 0, stream>>>(static_cast<const uint16_t*>(a.x), a.M, a.K, a.ldx,
                                                               reinterpret_cast<uint32_t*>(a.amax));
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t tiles = ((a.M + kFt - 1) / kFt) * ((a.K + kFt - 1) / kFt);
    const int grid2 = static_cast<int>(tiles < int64_t{sms} * 8 ? tiles : int64_t{sms} * 8);
    fp8_quantize_kernel<<<grid2, kFThreads, 0, stream>>>(static_cast<const uint16_t*>(a.x), a.M, a.K, a.ldx,
                                                         static_cast<uint8_t*>(a.q_row), a.ldr,
                                                         static_cast<uint8_t*>(a.q_col), a.ldc, a.amax, a.scale_inv);
    return cudaGetLastError();
}

}  // namespace mxfp4
