// launch_fp8.h -- host-side launch interface of the hybrid-backward FP8 kernels
// (quantize_fp8.cu, gemm_fp8.cu).  Internal to the library.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

namespace mxfp4 {

// Tensorwise E5M2 quantization of bf16 X[M,K] (row pitch ldx elements).  q_row: [M, ldr]
// codes of X, q_col: [K, ldc] codes of X^T (either may be null); ldr / ldc are the
// 16-byte-rounded row lengths.  amax and scale_inv: one fp32 each, device memory.
struct Fp8QuantArgs {
    const void* x;
    int64_t M, K, ldx;
    void* q_row;
    int64_t ldr;
    void* q_col;
    int64_t ldc;
    float* amax;
    float* scale_inv;
    int32_t amax_given;  // *amax already holds max |x|: no zeroing, no amax pass
};

// Up to kMaxFp8Tasks tensors in one pass of each kernel: row_end / tile_end are the
// running totals of each task's rows and 64 x 64 tiles.
constexpr int kMaxFp8Tasks = 4;
struct Fp8QuantBatch {
    Fp8QuantArgs t[kMaxFp8Tasks];
    int64_t row_end[kMaxFp8Tasks];
    int64_t tile_end[kMaxFp8Tasks];
    int32_t count;
    uint32_t* err;       // device error word (non-finite amax)
};

cudaError_t launch_fp8_quantize(const Fp8QuantBatch& b, int sms, cudaStream_t stream);

// One FP8 GEMM C[M,N] = (A . B^T) * (*a_scale_inv) * (*b_scale_inv): A [M, K] and B [N, K]
// E5M2 codes, K-major, row pitches lda / ldb bytes.
struct Fp8GemmArgs {
    int64_t M, N;
    int32_t tiles_m2;    // ceil(M / 256)
    int32_t tiles_n;     // ceil(N / 256)
    int32_t k_stages;    // ceil(K / 128): 128-element K steps
    void* c;
    int64_t ldc;
    int32_t out_f32;
    int32_t c_tma;
    const float* a_scale_inv;
    const float* b_scale_inv;
    uint32_t* err;
};

// Up to kMaxFp8Tasks GEMMs in one launch of CTA pairs, tile t belonging to the first
// problem j with t < tile_end[j].  amap / bmap: u8 {K, rows} maps, box {128, 128}, 128-byte
// swizzle; cmap as for the MXFP4 GEMMs (box of 64 bytes x 32 rows, 64-byte swizzle).
struct Fp8GemmBatch {
    CUtensorMap amap[kMaxFp8Tasks];
    CUtensorMap bmap[kMaxFp8Tasks];
    CUtensorMap cmap[kMaxFp8Tasks];
    Fp8GemmArgs args[kMaxFp8Tasks];
    int32_t tile_end[kMaxFp8Tasks];
    int32_t count;
};

size_t gemm_fp8_smem_bytes();
int gemm_fp8_max_clusters();
cudaError_t launch_gemm_fp8(const Fp8GemmBatch& b, int clusters, cudaStream_t stream);

}  // namespace mxfp4
