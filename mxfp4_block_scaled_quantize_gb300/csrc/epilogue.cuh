// epilogue.cuh -- output conversion shared by the two GEMM kernels.
//
// The optional bias follows `_forward_impl` of MXFP4ColumnParallelLinear /
// MXFP4RowParallelLinear in primus_turbo_mxfp4_local.py: the GEMM writes its output in the
// output dtype and the layer then adds the bf16 bias vector to every row (`output + bias`).
// Fused here, with the same two roundings: the fp32 accumulator is first rounded to the
// output dtype, then the bias is added in fp32 and the sum rounded to the output dtype
// again (for fp32 output the first rounding is the identity).
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

namespace mxfp4 {

__device__ __forceinline__ uint32_t pack_bf16x2(uint32_t lo_bits, uint32_t hi_bits) {
    __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(lo_bits), __uint_as_float(hi_bits));
    return *reinterpret_cast<uint32_t*>(&h);
}

// Eight bf16 bias values for output columns col .. col + 7 (zero past N).  Every lane of a
// warp asks for the same columns, so the load is one broadcast.  `bias` is 16-byte aligned
// and col is a multiple of 8.
__device__ __forceinline__ uint4 load_bias8(const uint16_t* bias, int64_t col, int64_t N) {
    if (col + 8 <= N) return __ldg(reinterpret_cast<const uint4*>(bias + col));
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t lo = col + 2 * i < N ? __ldg(bias + col + 2 * i) : 0u;
        const uint32_t hi = col + 2 * i + 1 < N ? __ldg(bias + col + 2 * i + 1) : 0u;
        w[i] = lo | (hi << 16);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ uint32_t uint4_word(const uint4& u, int i) {
    return i == 0 ? u.x : i == 1 ? u.y : i == 2 ? u.z : u.w;
}

// Two adjacent bf16 outputs with their bias pair (low half = even column).
__device__ __forceinline__ uint32_t pack_bf16x2_bias(uint32_t lo_bits, uint32_t hi_bits, uint32_t bias2) {
    const __nv_bfloat162 t = __floats2bfloat162_rn(__uint_as_float(lo_bits), __uint_as_float(hi_bits));
    const float2 tf = __bfloat1622float2(t);
    const float b0 = __uint_as_float(bias2 << 16);
    const float b1 = __uint_as_float(bias2 & 0xFFFF0000u);
    __nv_bfloat162 y = __floats2bfloat162_rn(__fadd_rn(tf.x, b0), __fadd_rn(tf.y, b1));
    return *reinterpret_cast<uint32_t*>(&y);
}

// One fp32 output plus the bf16 bias value in the low or high half of bias2.
__device__ __forceinline__ uint32_t add_bias_f32(uint32_t acc_bits, uint32_t bias2, int hi) {
    const float b = __uint_as_float(hi ? (bias2 & 0xFFFF0000u) : (bias2 << 16));
    return __float_as_uint(__fadd_rn(__uint_as_float(acc_bits), b));
}

// The 16 words of one 64-byte piece of an output row: 32 bf16 columns starting at v[0]
// (bf16 output) or 16 fp32 columns starting at v[0] (fp32 output); `col` is the piece's
// first output column.
template <bool kF32>
__device__ __forceinline__ void convert_piece(const uint32_t* v, const uint16_t* bias, int64_t col, int64_t N,
                                              uint32_t* w) {
    if (kF32) {
        if (bias == nullptr) {
#pragma unroll
            for (int i = 0; i < 16; ++i) w[i] = v[i];
        } else {
#pragma unroll
            for (int g8 = 0; g8 < 2; ++g8) {
                const uint4 bb = load_bias8(bias, col + 8 * g8, N);
#pragma unroll
                for (int i = 0; i < 8; ++i) w[8 * g8 + i] = add_bias_f32(v[8 * g8 + i], uint4_word(bb, i >> 1), i & 1);
            }
        }
    } else {
        if (bias == nullptr) {
#pragma unroll
            for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
        } else {
#pragma unroll
            for (int g8 = 0; g8 < 4; ++g8) {
                const uint4 bb = load_bias8(bias, col + 8 * g8, N);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    w[4 * g8 + i] = pack_bf16x2_bias(v[8 * g8 + 2 * i], v[8 * g8 + 2 * i + 1], uint4_word(bb, i));
            }
        }
    }
}

// One output element for the plain-store path.
__device__ __forceinline__ __nv_bfloat16 out_bf16(uint32_t acc_bits, const uint16_t* bias, int64_t col) {
    const __nv_bfloat16 t = __float2bfloat16_rn(__uint_as_float(acc_bits));
    if (bias == nullptr) return t;
    const float b = __uint_as_float(static_cast<uint32_t>(__ldg(bias + col)) << 16);
    return __float2bfloat16_rn(__fadd_rn(__bfloat162float(t), b));
}

__device__ __forceinline__ float out_f32(uint32_t acc_bits, const uint16_t* bias, int64_t col) {
    const float a = __uint_as_float(acc_bits);
    if (bias == nullptr) return a;
    return __fadd_rn(a, __uint_as_float(static_cast<uint32_t>(__ldg(bias + col)) << 16));
}

}  // namespace mxfp4
