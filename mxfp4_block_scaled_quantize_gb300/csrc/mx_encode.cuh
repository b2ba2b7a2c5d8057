// mx_encode.cuh -- the MX block arithmetic shared by the quantizer and the GEMM epilogue
// that quantizes its own output: the E8M0 scale byte of a 32-element block from its largest
// magnitude, max(expfield - 2, 0) (the OCP MX rule for E2M1, whose largest power of two is
// 2^2), and the E2M1 codes of the elements times 2^(127 - byte), rounded to nearest even and
// saturated at 6 by the hardware conversion.
#pragma once

#include <cstdint>

namespace mxfp4 {

// E8M0 byte of a block from the bf16 bit pattern of its largest magnitude (sign ignored):
// max(expfield - 2, 0).
__device__ __forceinline__ uint32_t scale_byte(uint32_t amax_bits) {
    const uint32_t ef = (amax_bits >> 7) & 0xFFu;
    return max(ef, 2u) - 2u;
}

// 2^(127 - byte) as fp32: always a normal number for byte in [0, 252].
__device__ __forceinline__ uint32_t inv_scale_bits(uint32_t byte) { return (254u - byte) << 23; }

// Magnitude-wise max of two bf16x2 words (the result's signs are not meaningful).
__device__ __forceinline__ uint32_t absmax2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint64_t pack2(uint32_t lo, uint32_t hi) {
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "r"(lo), "r"(hi));
    return d;
}

// Four words of consecutive bf16 pairs (elements 2k in the low half) times the scale pair
// `s2` -> four bytes of E2M1 codes, element 2k in the low nibble of byte k.
__device__ __forceinline__ uint32_t encode8(uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3,
                                            uint64_t s2) {
    uint32_t q;
    asm("{\n\t"
        ".reg .b32 l0, h0, l1, h1, l2, h2, l3, h3;\n\t"
        ".reg .b64 x0, x1, x2, x3;\n\t"
        ".reg .f32 a0, b0, a1, b1, a2, b2, a3, b3;\n\t"
        ".reg .b8 t0, t1, t2, t3;\n\t"
        "shl.b32 l0, %1, 16;\n\tand.b32 h0, %1, 0xFFFF0000;\n\t"
        "shl.b32 l1, %2, 16;\n\tand.b32 h1, %2, 0xFFFF0000;\n\t"
        "shl.b32 l2, %3, 16;\n\tand.b32 h2, %3, 0xFFFF0000;\n\t"
        "shl.b32 l3, %4, 16;\n\tand.b32 h3, %4, 0xFFFF0000;\n\t"
        "mov.b64 x0, {l0, h0};\n\tmov.b64 x1, {l1, h1};\n\t"
        "mov.b64 x2, {l2, h2};\n\tmov.b64 x3, {l3, h3};\n\t"
        "mul.rn.f32x2 x0, x0, %5;\n\tmul.rn.f32x2 x1, x1, %5;\n\t"
        "mul.rn.f32x2 x2, x2, %5;\n\tmul.rn.f32x2 x3, x3, %5;\n\t"
        "mov.b64 {a0, b0}, x0;\n\tmov.b64 {a1, b1}, x1;\n\t"
        "mov.b64 {a2, b2}, x2;\n\tmov.b64 {a3, b3}, x3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t0, b0, a0;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t1, b1, a1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t2, b2, a2;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t3, b3, a3;\n\t"
        "mov.b32 %0, {t0, t1, t2, t3};\n\t}"
        : "=r"(q)
        : "r"(w0), "r"(w1), "r"(w2), "r"(w3), "l"(s2));
    return q;
}

}  // namespace mxfp4
