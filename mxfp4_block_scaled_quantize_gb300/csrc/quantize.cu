// quantize.cu -- MXFP4 row-only and dual (row + column) quantizer for sm_103a.
//
// What it computes (primus_turbo_mxfp4_local.py, `_quantize_mxfp4_dual_op` with all
// recipe and shuffle flags off, shapes per `_quantize_mxfp4_dual_fake`; the row-only
// variant is the "row-only packing" of Primus PR #1107): for every 32-element block of
// bf16 values, along K for the row blob and along M for the column blob, the E8M0 scale
// byte max(expfield(amax) - 2, 0) -- which is floor(log2 amax) - 2 clamped at -127, read
// off the bf16 exponent bits (a subnormal or zero amax has exponent field 0 and gets the
// clamped byte 0) -- and the E2M1 codes of v * 2^(127 - byte), rounded to nearest even and
// saturated at 6 by the hardware conversion.  The power-of-two scaling is exact in fp32.
//
// Design: a persistent grid, one 128 x 128 bf16 tile (32 KB) per step.  One producer
// thread streams tiles into a 3-stage shared-memory ring with TMA, as two 64-column boxes
// with the 128-byte swizzle (out-of-bounds rows and columns arrive as zeros, which is
// exactly the padding rule).  8 consumer warps quantize each tile twice from shared
// memory, so X is read from HBM once for both packings:
//   rowwise     one thread per 32-element block: four 16-byte reads, an abs-max tree of
//               packed bf16 maxima, 16 packed fp32x2 multiplies, 16 conversions, one
//               16-byte store of the codes; a warp covers 16 whole rows, so its stores are
//               whole 32-byte sectors;
//   columnwise  one thread per column pair of a 32-row block: 32 4-byte reads, the same
//               abs-max and conversions with the pair's two scales in one fp32x2 multiply;
//               a warp covers 8 column pairs and all four row blocks, so each store
//               instruction writes 64-byte runs of 8 column-blob rows.
// (Measured on GB300: whole-sector stores took the dY quantization of the Flux MLP step
// from 35.4 to 30.7 us.)  The swizzle makes both access patterns bank-conflict free.
// Consumer warps never wait
// for each other (except for 2-D blocks, below): each warp waits for the stage itself,
// stores its codes and scale bytes straight to global memory, and releases the stage with
// its own barrier arrival.
//
// 2-D blocks (the weight recipe of `_quantize_weight_dual`, `rowwise_use_2d_block` and
// `colwise_use_2d_block`): X is cut into 32 x 32 blocks, each gets one scale byte from the
// amax of its 1024 elements by the same rule, and both packings encode every element of the
// block with it.  A 128 x 128 tile holds 16 whole blocks: each rowwise thread's 1 x 32 amax
// is folded over the 4 lanes of its warp that share the block and written per warp to
// shared memory; after one named barrier of the consumer warps every thread takes the
// block's maximum over the 8 warps, for its row blocks and, in the columnwise pass, for
// its column pair (both columns lie in one block).  Scale bytes of padding rows of the
// tensor-core layout stay 0x00, as in the 1-D packings.
//
// Hadamard transform of the column blob (the `colwise_use_rht` flag of the activation and
// gradient quantizers): before the columnwise pass quantizes a column, each group of 16
// consecutive rows becomes (1/4) H16 diag(s) of itself, s a sign mask of the task, computed
// in fp32 -- signs, butterflies for h = 1, 2, 4, 8, then x 0.25 -- and the 32-row MX block is
// quantized from these fp32 values.  For such a task a warp takes one 32-row block and 32
// consecutive column pairs, so its shared reads are whole tile rows, conflict free in
// natural row order, and each thread's registers hold its rows in order: the butterflies
// are plain register pairs, with the difference taken lower minus upper row as the
// definition has it.
#include <cuda_bf16.h>

#include "launch.h"
#include "mx_encode.cuh"
#include "ptx.cuh"

namespace mxfp4 {
namespace {

constexpr int kQT = 128;                       // tile edge (rows and columns)
constexpr int kQStages = 3;
constexpr int kQConsumerWarps = 8;
constexpr int kQConsumers = kQConsumerWarps * 32;
constexpr int kQThreads = kQConsumers + 32;    // + one producer warp
constexpr int kQTileBytes = kQT * kQT * 2;
constexpr int kQCtasPerSm = 2;   // 18 warps: 96 registers per thread (a sub-partition holds 5 warps)

struct QuantSmem {
    uint8_t tile[kQStages][kQTileBytes];       // per stage: two 64-column swizzled boxes
    uint64_t full[kQStages];
    uint64_t empty[kQStages];                  // one arrival per consumer warp
    // 2-D blocks: per tile parity, per consumer warp, per block (row group Q, block column
    // b): the warp's largest magnitude (bf16 bits) in that block
    uint32_t part[2][kQConsumerWarps][16];
    int abort;
};
constexpr uint32_t kBarConsumers = 1;          // named barrier of the consumer warps

constexpr int kQBoxBytes = kQT * 128;          // 128 rows x 64 bf16 columns

// Byte offset of (row r, 16-byte chunk j of the 128-byte box row) under the 128-byte
// swizzle: chunk j of row r is stored at chunk j ^ (r % 8).
__device__ __forceinline__ uint32_t swz(int r, int j) { return r * 128 + ((j ^ (r & 7)) << 4); }

// Eight words = rows 2j, 2j+1 (j = 0..3) of a column pair (column c0 in the low halves,
// c1 in the high halves), times the pair's scales `s2` = {s(c0), s(c1)}: four bytes of
// codes for c0 (*q0) and for c1 (*q1), row 2j in the low nibble of byte j.
__device__ __forceinline__ void encode_cols8(const uint32_t* w, uint64_t s2, uint32_t* q0,
                                             uint32_t* q1) {
    asm("{\n\t"
        ".reg .b32 l<8>, h<8>;\n\t"
        ".reg .b64 x<8>;\n\t"
        ".reg .f32 a<8>, b<8>;\n\t"
        ".reg .b8 c<4>, d<4>;\n\t"
        "shl.b32 l0, %2, 16;\n\tand.b32 h0, %2, 0xFFFF0000;\n\t"
        "shl.b32 l1, %3, 16;\n\tand.b32 h1, %3, 0xFFFF0000;\n\t"
        "shl.b32 l2, %4, 16;\n\tand.b32 h2, %4, 0xFFFF0000;\n\t"
        "shl.b32 l3, %5, 16;\n\tand.b32 h3, %5, 0xFFFF0000;\n\t"
        "shl.b32 l4, %6, 16;\n\tand.b32 h4, %6, 0xFFFF0000;\n\t"
        "shl.b32 l5, %7, 16;\n\tand.b32 h5, %7, 0xFFFF0000;\n\t"
        "shl.b32 l6, %8, 16;\n\tand.b32 h6, %8, 0xFFFF0000;\n\t"
        "shl.b32 l7, %9, 16;\n\tand.b32 h7, %9, 0xFFFF0000;\n\t"
        "mov.b64 x0, {l0, h0};\n\tmov.b64 x1, {l1, h1};\n\t"
        "mov.b64 x2, {l2, h2};\n\tmov.b64 x3, {l3, h3};\n\t"
        "mov.b64 x4, {l4, h4};\n\tmov.b64 x5, {l5, h5};\n\t"
        "mov.b64 x6, {l6, h6};\n\tmov.b64 x7, {l7, h7};\n\t"
        "mul.rn.f32x2 x0, x0, %10;\n\tmul.rn.f32x2 x1, x1, %10;\n\t"
        "mul.rn.f32x2 x2, x2, %10;\n\tmul.rn.f32x2 x3, x3, %10;\n\t"
        "mul.rn.f32x2 x4, x4, %10;\n\tmul.rn.f32x2 x5, x5, %10;\n\t"
        "mul.rn.f32x2 x6, x6, %10;\n\tmul.rn.f32x2 x7, x7, %10;\n\t"
        "mov.b64 {a0, b0}, x0;\n\tmov.b64 {a1, b1}, x1;\n\t"
        "mov.b64 {a2, b2}, x2;\n\tmov.b64 {a3, b3}, x3;\n\t"
        "mov.b64 {a4, b4}, x4;\n\tmov.b64 {a5, b5}, x5;\n\t"
        "mov.b64 {a6, b6}, x6;\n\tmov.b64 {a7, b7}, x7;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 c0, a1, a0;\n\tcvt.rn.satfinite.e2m1x2.f32 d0, b1, b0;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 c1, a3, a2;\n\tcvt.rn.satfinite.e2m1x2.f32 d1, b3, b2;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 c2, a5, a4;\n\tcvt.rn.satfinite.e2m1x2.f32 d2, b5, b4;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 c3, a7, a6;\n\tcvt.rn.satfinite.e2m1x2.f32 d3, b7, b6;\n\t"
        "mov.b32 %0, {c0, c1, c2, c3};\n\t"
        "mov.b32 %1, {d0, d1, d2, d3};\n\t}"
        : "=r"(*q0), "=r"(*q1)
        : "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7]),
          "l"(s2));
}

// ---- stochastic rounding of the elements (the gradient quantizer's `use_sr` flag) -------
// Random bits: Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC 2011), key = the 64-bit seed,
// counter = (b / 8, a, packing, 0) for blob row a, blob column b (packing 0: row blob of
// X; 1: col blob, whose row a is column a of X); word (b / 2) % 4 of the result carries
// the element's 16 bits, in its low half for even b.  One call serves 8 consecutive
// elements of a blob row.
__device__ __forceinline__ uint4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint64_t seed) {
    uint32_t x0 = c0, x1 = c1, x2 = c2, x3 = 0u;
    uint32_t k0 = static_cast<uint32_t>(seed), k1 = static_cast<uint32_t>(seed >> 32);
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        uint64_t p0, p1;   // full 64-bit products, one wide multiply each
        asm("mul.wide.u32 %0, %1, 0xD2511F53;" : "=l"(p0) : "r"(x0));
        asm("mul.wide.u32 %0, %1, 0xCD9E8D57;" : "=l"(p1) : "r"(x2));
        const uint32_t hi0 = static_cast<uint32_t>(p0 >> 32), lo0 = static_cast<uint32_t>(p0);
        const uint32_t hi1 = static_cast<uint32_t>(p1 >> 32), lo1 = static_cast<uint32_t>(p1);
        const uint32_t n0 = hi1 ^ x1 ^ k0, n2 = hi0 ^ x3 ^ k1;
        x0 = n0;
        x1 = lo1;
        x2 = n2;
        x3 = lo0;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return make_uint4(x0, x1, x2, x3);
}

// Stochastic rounding of one element onto the E2M1 magnitudes {0, .5, 1, 1.5, 2, 3, 4, 6}:
// a = |y| (y the scaled element, |y| < 8 for a finite block), x: a value with y's sign bit,
// r: 16 random bits.  |y| >= 6 gives 6; otherwise, between neighbours lo <= |y| < hi, hi
// when r is below t = floor((|y| - lo) / g * 2^16) (g = hi - lo), else lo; the sign is kept.
// Computed as floor_g(|y| + g * (65535 - r) / 2^16), which reaches hi exactly when t > r.  g
// is 0.5 below 2, 1 in [2, 4) and 2 in [4, 8).  Two fp32 adds rounded toward zero do it:
// s1 = |y| + g * (1 + (65535 - r) / 2^16), whose second operand is built from bits, then
// s1 + g * 2^23, where the fp32 spacing is g, so the sum is g * 2^23 + floor_g(s1);
// subtracting g * 2^23 + g leaves floor_g(|y| + noise).  Rounding s1 toward zero keeps its
// floor on the g grid (a multiple of s1's own spacing).  A result of 8 (|y| in [6, 8)) is
// left to the saturating conversion, which gives 6.
__device__ __forceinline__ float sr_round(float a, float x, uint32_t r) {
    const uint32_t e = max(__float_as_uint(a) >> 23, 127u);
    const uint32_t gbits = (e - 1u) << 23;                               // g = 2^(e - 128)
    const float noise = __uint_as_float(gbits | ((r ^ 0xFFFFu) << 7));   // g * (1 + (65535 - r) / 2^16)
    const uint32_t cbits = gbits + (23u << 23);                          // g * 2^23
    const float s2 = __fadd_rz(__fadd_rz(a, noise), __uint_as_float(cbits));
    const float q = __fsub_rn(s2, __uint_as_float(cbits + 1u));          // - (g * 2^23 + g)
    return __uint_as_float(__float_as_uint(q) | (__float_as_uint(x) & 0x80000000u));
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t rnd16(uint32_t w, int hi) { return hi ? (w >> 16) : (w & 0xFFFFu); }

// Eight grid values -> four bytes of codes, element 2k in the low nibble of byte k.
__device__ __forceinline__ uint32_t pack_e2m1x8(const float* f) {
    uint32_t q;
    asm("{\n\t.reg .b8 t0, t1, t2, t3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t3, %8, %7;\n\t"
        "mov.b32 %0, {t0, t1, t2, t3};\n\t}"
        : "=r"(q)
        : "f"(f[0]), "f"(f[1]), "f"(f[2]), "f"(f[3]), "f"(f[4]), "f"(f[5]), "f"(f[6]), "f"(f[7]));
    return q;
}

// encode8 with stochastic rounding: 8 consecutive elements of a blob row (v: word k holds
// elements 2k, 2k+1), their scale 2^(127 - byte) as fp32, and their Philox words.
__device__ __forceinline__ uint32_t encode8_sr(uint4 v, float inv, uint4 rw) {
    const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
    const uint32_t r4[4] = {rw.x, rw.y, rw.z, rw.w};
    float f[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const float x = (e & 1) ? bf16_hi(vw[e >> 1]) : bf16_lo(vw[e >> 1]);
        f[e] = sr_round(__fmul_rn(fabsf(x), inv), x, rnd16(r4[e >> 1], e & 1));
    }
    return pack_e2m1x8(f);
}

// The Philox words of an 8-row group of the column pass in register order: register k of
// the group holds row k ^ 2rb, whose bits are in word (k / 2) ^ rb of the true order.
__device__ __forceinline__ void words_in_register_order(uint4 r, uint32_t rb, uint32_t* o) {
    uint32_t a0 = r.x, a1 = r.y, a2 = r.z, a3 = r.w;
    if (rb & 1u) {
        uint32_t t = a0; a0 = a1; a1 = t; t = a2; a2 = a3; a3 = t;
    }
    if (rb & 2u) {
        uint32_t t = a0; a0 = a2; a2 = t; t = a1; a1 = a3; a3 = t;
    }
    o[0] = a0; o[1] = a1; o[2] = a2; o[3] = a3;
}

// encode_cols8 with stochastic rounding.  w[k] holds rows (k ^ 2rb) of the 8-row group
// (column c0 in the low halves, c1 in the high halves); r0 / r1: the Philox words of the
// group's 8 rows for c0 / c1, in true row order.  Output bytes in w's (permuted) order, as
// encode_cols8 gives them.
__device__ __forceinline__ void encode_cols8_sr(const uint32_t* w, float inv0, float inv1, uint4 r0, uint4 r1,
                                                uint32_t rb, uint32_t* q0, uint32_t* q1) {
    uint32_t ra[4], rbw[4];
    words_in_register_order(r0, rb, ra);
    words_in_register_order(r1, rb, rbw);
    float f0[8], f1[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const float x0 = bf16_lo(w[k]), x1 = bf16_hi(w[k]);
        f0[k] = sr_round(__fmul_rn(fabsf(x0), inv0), x0, rnd16(ra[k >> 1], k & 1));
        f1[k] = sr_round(__fmul_rn(fabsf(x1), inv1), x1, rnd16(rbw[k >> 1], k & 1));
    }
    *q0 = pack_e2m1x8(f0);
    *q1 = pack_e2m1x8(f1);
}

__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ float lo_f(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v)); }
__device__ __forceinline__ float hi_f(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v >> 32)); }

// The Hadamard transform of the two columns of a column pair over one 32-row block, register
// i of w holding row i (column c0 in the low halves, c1 in the high halves); bit j of
// `signs` negates row j of each 16-row group.  Both columns go through every fp32 step
// together as pairs (packed adds, subtractions and multiplies, each rounding to nearest
// even per lane, so each column gets exactly its own sequence).  Gives the two blocks'
// scale bytes from the transformed values and their codes, word g byte j holding rows
// 8g + 2j (low nibble) and 8g + 2j + 1.  kSR: the scaled transformed elements are
// stochastically rounded with the col-blob bits of Philox counter (c0 + g, a + column, 1, 0)
// for row group g (c0: the block's first row / 8, a: the pair's first column).
template <bool kSR>
__device__ __forceinline__ void rht_pair(const uint32_t* w, uint32_t signs, uint32_t* byte0, uint32_t* byte1,
                                         uint32_t* q0, uint32_t* q1, uint64_t seed, uint32_t c0, uint32_t a) {
    uint64_t f[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const uint32_t sb = ((signs >> (i & 15)) & 1u) << 31;
        f[i] = pack2((w[i] << 16) ^ sb, (w[i] & 0xFFFF0000u) ^ sb);
    }
#pragma unroll
    for (int g = 0; g < 32; g += 16) {
#pragma unroll
        for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                if (i & h) continue;
                const uint64_t lo = f[g + i], hi = f[g + i + h];
                f[g + i] = add2(lo, hi);
                f[g + i + h] = sub2(lo, hi);
            }
        }
    }
    const uint64_t quarter = pack2(0x3E800000u, 0x3E800000u);   // 0.25
    float m0 = 0.0f, m1 = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        f[i] = mul2(f[i], quarter);
        m0 = fmaxf(m0, fabsf(lo_f(f[i])));
        m1 = fmaxf(m1, fabsf(hi_f(f[i])));
    }
    // floor(log2) + 127 of a normal amax
    const uint32_t b0 = max((__float_as_uint(m0) >> 23) & 0xFFu, 2u) - 2u;
    const uint32_t b1 = max((__float_as_uint(m1) >> 23) & 0xFFu, 2u) - 2u;
    *byte0 = b0;
    *byte1 = b1;
    float g0[8], g1[8];
    if (kSR) {
        const float inv0 = __uint_as_float(inv_scale_bits(b0)), inv1 = __uint_as_float(inv_scale_bits(b1));
#pragma unroll
        for (int gw = 0; gw < 4; ++gw) {
            const uint4 r0 = philox4x32_10(c0 + gw, a, 1u, seed);
            const uint4 r1 = philox4x32_10(c0 + gw, a + 1u, 1u, seed);
            const uint32_t p0[4] = {r0.x, r0.y, r0.z, r0.w}, p1[4] = {r1.x, r1.y, r1.z, r1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float y0 = lo_f(f[8 * gw + i]), y1 = hi_f(f[8 * gw + i]);
                g0[i] = sr_round(__fmul_rn(fabsf(y0), inv0), y0, rnd16(p0[i >> 1], i & 1));
                g1[i] = sr_round(__fmul_rn(fabsf(y1), inv1), y1, rnd16(p1[i >> 1], i & 1));
            }
            q0[gw] = pack_e2m1x8(g0);
            q1[gw] = pack_e2m1x8(g1);
        }
    } else {
        const uint64_t inv2 = pack2(inv_scale_bits(b0), inv_scale_bits(b1));
#pragma unroll
        for (int gw = 0; gw < 4; ++gw) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint64_t y = mul2(f[8 * gw + i], inv2);
                g0[i] = lo_f(y);
                g1[i] = hi_f(y);
            }
            q0[gw] = pack_e2m1x8(g0);
            q1[gw] = pack_e2m1x8(g1);
        }
    }
}

__device__ __forceinline__ uint32_t lds32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}

__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(a));
    return v;
}

// kRecipes: some task of the launch has 2-D blocks (QuantArgs::block_2d) or the Hadamard
// transform of its column blob (QuantArgs::rht); such a task's tiles take those paths.
// The stochastic-rounding instance runs one CTA per SM, with the registers that leaves a
// thread: at two CTAs per SM (96 registers) its Philox words spilled.
template <bool kDual, bool kSR, bool kRecipes>
__global__ void __launch_bounds__(kQThreads, kSR ? 1 : kQCtasPerSm)
    quantize_kernel(const __grid_constant__ QuantBatch P) {
    extern __shared__ uint8_t smem_raw[];
    QuantSmem& sm = *reinterpret_cast<QuantSmem*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int num_tiles = P.tile_end[P.count - 1];
    uint32_t* const err = P.args[0].err;
    // Task of launch tile t, and t's index within that task.
    auto task_of = [&](int t, int* local) {
        int j = 0;
        while (j + 1 < P.count && t >= P.tile_end[j]) ++j;
        *local = t - (j > 0 ? P.tile_end[j - 1] : 0);
        return j;
    };

    if (tid == 0) {
        for (int s = 0; s < kQStages; ++s) {
            mbar_init(smem_addr(&sm.full[s]), 1);
            mbar_init(smem_addr(&sm.empty[s]), kQConsumerWarps);
        }
        sm.abort = 0;
        fence_barrier_init();
    }
    __syncthreads();
    grid_launch_dependents();
    grid_wait_prerequisites();

    if (warp == kQConsumerWarps) {
        // ------------------------------------------------------------- producer (TMA)
        if (lane_id() == 0) {
            for (int j = 0; j < P.count; ++j) prefetch_tensormap(&P.maps[j]);
            int it = 0;
            for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++it) {
                const int s = it % kQStages;
                const uint32_t ph = (it / kQStages) & 1;
                if (!mbar_wait(smem_addr(&sm.empty[s]), ph ^ 1, err, kErrQuantProducer, &sm.abort))
                    break;
                int lt;
                const int j = task_of(t, &lt);
                const int tm = lt / P.args[j].tiles_k, tk = lt % P.args[j].tiles_k;
                const CUtensorMap* xmap = &P.maps[j];
                const uint32_t bar = smem_addr(&sm.full[s]);
                mbar_arrive_expect_tx(bar, kQTileBytes);
                tma_load_2d(smem_addr(sm.tile[s]), xmap, tk * kQT, tm * kQT, bar);
                tma_load_2d(smem_addr(sm.tile[s]) + kQBoxBytes, xmap, tk * kQT + 64, tm * kQT, bar);
            }
            // Drain: every armed stage's copy has landed before this thread may leave.
            const int armed = it < kQStages ? it : kQStages;
            for (int i = 1; i <= armed; ++i) {
                const int j = it - i;
                mbar_wait_quiet(smem_addr(&sm.full[j % kQStages]), (j / kQStages) & 1, kWaitLimitNs);
            }
        }
        return;
    }

    // ------------------------------------------------------------------ consumers
    const uint32_t lane = lane_id();
    uint32_t amx[kMaxQuantTasks] = {0u, 0u, 0u, 0u};   // row-only: per task, this lane's max |x| so far
    int it = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++it) {
        const int s = it % kQStages;
        const uint32_t ph = (it / kQStages) & 1;
        int ok = 0;
        if (lane == 0) ok = mbar_wait(smem_addr(&sm.full[s]), ph, err, kErrQuantConsumer, &sm.abort) ? 1 : 0;
        if (!__shfl_sync(0xFFFFFFFFu, ok, 0)) break;

        int lt;
        const int pj = task_of(t, &lt);
        const QuantArgs& p = P.args[pj];
        const int tm = lt / p.tiles_k, tk = lt % p.tiles_k;
        const int64_t m0 = static_cast<int64_t>(tm) * kQT;
        const int64_t k0 = static_cast<int64_t>(tk) * kQT;
        const uint32_t tile = smem_addr(sm.tile[s]);
        // Tensor-core layout: this tile's scales are exactly one 512-byte atom per packing.
        uint8_t* const atom_row = p.s_row + (static_cast<int64_t>(tm) * (p.kb_row >> 2) + tk) * 512;
        uint8_t* const atom_col = kDual ? p.s_col + (static_cast<int64_t>(tk) * (p.kb_col >> 2) + tm) * 512 : nullptr;

        // ---- rowwise: one thread per 32-element block.  Warp w takes atom lines
        //      L = 4w..4w+3 (rows L, L+32, L+64, L+96) and all four block columns, so each
        //      store instruction writes whole 32-byte sectors of 16 rows, and each quarter
        //      warp's 16-byte shared reads hit 8 distinct swizzled chunks.
        const bool blk2d = kRecipes && p.block_2d;
        const int L = 4 * warp + (lane & 3);
        const int Q = lane >> 3;
        const int r = Q * 32 + L;
        const int64_t row = m0 + r;
        uint4 v[2][4];
        uint32_t bm[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int b = ((lane >> 2) & 1) + 2 * i;
            const uint32_t box = tile + (b >> 1) * kQBoxBytes;
            const int j0 = (b & 1) * 4;
#pragma unroll
            for (int c = 0; c < 4; ++c) v[i][c] = lds128(box + swz(r, j0 + c));
            uint32_t m = absmax2(absmax2(absmax2(v[i][0].x, v[i][0].y), absmax2(v[i][0].z, v[i][0].w)),
                                 absmax2(absmax2(v[i][1].x, v[i][1].y), absmax2(v[i][1].z, v[i][1].w)));
            m = absmax2(m, absmax2(absmax2(absmax2(v[i][2].x, v[i][2].y), absmax2(v[i][2].z, v[i][2].w)),
                                   absmax2(absmax2(v[i][3].x, v[i][3].y), absmax2(v[i][3].z, v[i][3].w))));
            m = absmax2(m, m >> 16) & 0x7FFFu;   // the block's largest magnitude, bf16 bits
            bm[i] = m;
        }
        const int par = it & 1;
        if (blk2d) {
            // fold over the 4 lanes of the warp that share (Q, b), then one word per warp
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                bm[i] = max(bm[i], __shfl_xor_sync(0xFFFFFFFFu, bm[i], 1));
                bm[i] = max(bm[i], __shfl_xor_sync(0xFFFFFFFFu, bm[i], 2));
                if ((lane & 3) == 0) sm.part[par][warp][Q * 4 + ((lane >> 2) & 1) + 2 * i] = bm[i];
            }
            named_barrier(kBarConsumers, kQConsumers);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int b = ((lane >> 2) & 1) + 2 * i;
                uint32_t m = 0;
#pragma unroll
                for (int w = 0; w < kQConsumerWarps; ++w) m = max(m, sm.part[par][w][Q * 4 + b]);
                bm[i] = m;
            }
        }
        if (!kDual && p.amax_bits != nullptr) {   // running max |x| per task, folded in once at exit
            const uint32_t m2 = max(bm[0], bm[1]);
#pragma unroll
            for (int k = 0; k < kMaxQuantTasks; ++k)
                if (k == pj) amx[k] = max(amx[k], m2);
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int b = ((lane >> 2) & 1) + 2 * i;
            const uint32_t byte = scale_byte(bm[i]);
            const uint32_t inv = inv_scale_bits(byte);
            uint4 q;
            if (kSR) {
                const float invf = __uint_as_float(inv);
                const uint32_t c0 = static_cast<uint32_t>((k0 + 32 * b) >> 3), a = static_cast<uint32_t>(row);
                q = make_uint4(encode8_sr(v[i][0], invf, philox4x32_10(c0 + 0, a, 0u, p.seed)),
                               encode8_sr(v[i][1], invf, philox4x32_10(c0 + 1, a, 0u, p.seed)),
                               encode8_sr(v[i][2], invf, philox4x32_10(c0 + 2, a, 0u, p.seed)),
                               encode8_sr(v[i][3], invf, philox4x32_10(c0 + 3, a, 0u, p.seed)));
            } else {
                const uint64_t s2 = pack2(inv, inv);
                q = make_uint4(encode8(v[i][0].x, v[i][0].y, v[i][0].z, v[i][0].w, s2),
                               encode8(v[i][1].x, v[i][1].y, v[i][1].z, v[i][1].w, s2),
                               encode8(v[i][2].x, v[i][2].y, v[i][2].z, v[i][2].w, s2),
                               encode8(v[i][3].x, v[i][3].y, v[i][3].z, v[i][3].w, s2));
            }
            if (row < p.M) {
                *reinterpret_cast<uint4*>(p.q_row + row * p.ldq_row + ((k0 + 32 * b) >> 1)) = q;
                if (!p.tc_layout) p.s_row[row * p.kb_row + (k0 >> 5) + b] = static_cast<uint8_t>(byte);
            }
            // Padding rows of the tensor-core layout get the byte 0x00 (a 1-D padding
            // block's own amax is 0; a 2-D block's rows past M do not carry its scale).
            if (p.tc_layout) atom_row[L * 16 + Q * 4 + b] = static_cast<uint8_t>(row < p.M ? byte : 0u);
        }

        // ---- columnwise: thread owns columns (2pc, 2pc+1) of the 32-row block rb; a warp
        //      takes 8 column pairs and all four row blocks, so each store instruction
        //      writes the whole 64-byte run of 8 column-blob rows.  Row block rb walks its
        //      rows in the order i ^ 2rb, which puts the four quarter warps of every shared
        //      read on four disjoint bank groups; the code bytes come out permuted by
        //      XOR rb and one byte permute puts them back.
        if (kDual) {
            // A task with the transform maps threads differently: warp w takes row block
            // w % 4 and 32 consecutive column pairs, so each shared read is one whole tile row
            // (conflict free in natural row order) and the butterflies pair registers the way
            // they pair rows.
            const bool rht_task = kRecipes && p.rht;
            const int pc = rht_task ? 32 * (warp >> 2) + lane : 8 * warp + (lane & 7);
            const int rb = rht_task ? (warp & 3) : (lane >> 3);
            const int xo = rht_task ? 0 : 2 * rb;   // register k of an 8-row group holds row k ^ xo
            const uint32_t box = tile + (pc >> 5) * kQBoxBytes;
            const int jc = (pc & 31) >> 2;
            const uint32_t inner = (pc & 3) * 4;
            // Offsets of rows (k ^ xo), k = 0..7, of each 8-row group; the group offset is a
            // compile-time constant of every load.
            uint32_t toff[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int rr = k ^ xo;
                toff[k] = box + rb * 32 * 128 + rr * 128 + ((jc ^ rr) << 4) + inner;
            }
            uint32_t w[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) w[i] = lds32(toff[i & 7] + (i & ~7) * 128);
            const uint32_t sel = 0x3210u ^ (0x1111u * static_cast<uint32_t>(xo >> 1));
            const int64_t kc = k0 + 2 * pc;
            uint32_t byte0, byte1;
            uint32_t q0[4], q1[4];
            if (rht_task) {
                // natural row order: register i holds row i of the block
                const uint32_t c0 = static_cast<uint32_t>((m0 + rb * 32) >> 3);
                rht_pair<kSR>(w, p.rht_signs, &byte0, &byte1, q0, q1, p.seed, c0, static_cast<uint32_t>(kc));
            } else {
            if (blk2d) {
                // both columns lie in block column pc / 16 of row group rb
                uint32_t m = 0;
#pragma unroll
                for (int w2 = 0; w2 < kQConsumerWarps; ++w2) m = max(m, sm.part[par][w2][rb * 4 + (pc >> 4)]);
                byte0 = byte1 = scale_byte(m);
            } else {
                uint32_t m = w[0];
#pragma unroll
                for (int i = 1; i < 32; ++i) m = absmax2(m, w[i]);
                byte0 = scale_byte(m);
                byte1 = scale_byte(m >> 16);
            }
            const uint64_t s2 = pack2(inv_scale_bits(byte0), inv_scale_bits(byte1));
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (kSR) {
                    const uint32_t c0 = static_cast<uint32_t>(((m0 + rb * 32) >> 3) + j);
                    encode_cols8_sr(&w[8 * j], __uint_as_float(inv_scale_bits(byte0)),
                                    __uint_as_float(inv_scale_bits(byte1)),
                                    philox4x32_10(c0, static_cast<uint32_t>(kc), 1u, p.seed),
                                    philox4x32_10(c0, static_cast<uint32_t>(kc + 1), 1u, p.seed),
                                    static_cast<uint32_t>(rb), &q0[j], &q1[j]);
                } else {
                    encode_cols8(&w[8 * j], s2, &q0[j], &q1[j]);
                }
                q0[j] = __byte_perm(q0[j], 0, sel);
                q1[j] = __byte_perm(q1[j], 0, sel);
            }
            }
            const int64_t off = (m0 + rb * 32) >> 1;
            if (kc < p.K) {
                *reinterpret_cast<uint4*>(p.q_col + kc * p.ldq_col + off) = make_uint4(q0[0], q0[1], q0[2], q0[3]);
                if (!p.tc_layout) p.s_col[kc * p.kb_col + (m0 >> 5) + rb] = static_cast<uint8_t>(byte0);
            }
            if (kc + 1 < p.K) {
                *reinterpret_cast<uint4*>(p.q_col + (kc + 1) * p.ldq_col + off) =
                    make_uint4(q1[0], q1[1], q1[2], q1[3]);
                if (!p.tc_layout) p.s_col[(kc + 1) * p.kb_col + (m0 >> 5) + rb] = static_cast<uint8_t>(byte1);
            }
            const int kl0 = 2 * pc, kl1 = 2 * pc + 1;
            if (p.tc_layout) {   // padding rows (columns of X past K) keep 0x00
                atom_col[(kl0 & 31) * 16 + (kl0 >> 5) * 4 + rb] = static_cast<uint8_t>(kc < p.K ? byte0 : 0u);
                atom_col[(kl1 & 31) * 16 + (kl1 >> 5) * 4 + rb] = static_cast<uint8_t>(kc + 1 < p.K ? byte1 : 0u);
            }
        }

        // This warp is done with the stage.
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&sm.empty[s]));
    }
    // The tasks' max |x| (bf16 magnitude bits -> fp32 bits): one atomic per warp and task.
#pragma unroll
    for (int k = 0; k < kMaxQuantTasks; ++k) {
        if (kDual || k >= P.count || P.args[k].amax_bits == nullptr) continue;
        const uint32_t m2 = __reduce_max_sync(0xFFFFFFFFu, amx[k]);
        if (lane == 0 && m2 != 0) atomicMax(P.args[k].amax_bits, m2 << 16);
    }
}

// ---- the quantizer prologue: QK RMSNorm + interleaved RoPE backward ------------------
// d(mixed_qkv) of the QKV projection computed in the staging read and quantized, instead of
// the norm + RoPE backward writing it to HBM for the quantizer to read back.  With head
// dimension 128 every 128-column tile of d(mixed_qkv) [M, H*3*128] is one (head, part):
// part 0 = q, 1 = k (computed), 2 = v (the gradient itself).  A CTA takes units of `span`
// consecutive tiles of one 128-row block, so each thread loads the RoPE cosines and sines
// of its row and columns once per unit into registers.  For a q / k tile the producer
// brings the gradient tile g and the tile of mixed_qkv x; each row's two rowwise threads
// (64 columns each) compute, in fp32, dy = the inverse rotation of g on the pairs
// (2i, 2i+1) (dy0 = g0 c + g1 s, dy1 = g1 c - g0 s), dn = dy w and their share of
// sum(dn x); the row's sum over both comes with one shuffle; a second pass recomputes dn and
// gives dx = r dn - (r^3 / 128) x sum(dn x), rounded to bf16 (to nearest even).  That bf16
// dx is what gets quantized: by the rowwise pass, and, written back over g in the stage, by
// the columnwise pass after a barrier of the consumer warps.  One CTA per SM (two 32 KB
// tiles per stage).

struct NormRopeSmem {
    uint8_t tile[kQStages][kQTileBytes];   // g, overwritten by dx for q / k tiles
    uint8_t xt[kQStages][kQTileBytes];     // mixed_qkv
    uint64_t full[kQStages];
    uint64_t empty[kQStages];
    float w[2][kNormRopeD];
    float rs[kQT][kNormRopeMaxUnitHeads * 2];   // the unit's saved r of each row, (head, part)
    int abort;
};

__device__ __forceinline__ void sts128q(uint32_t a, const uint4& v) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ uint32_t word_of(const uint4& u, int e) {
    return e == 0 ? u.x : e == 1 ? u.y : e == 2 ? u.z : u.w;
}

// dn = (the inverse rotation of the 8 gradient elements in gw) * w for columns kk .. kk + 7
// of a head (kk a multiple of 8), with the row's cosines / sines of pairs kk/2 .. kk/2 + 3.
__device__ __forceinline__ void norm_rope_dn(const uint4& gw, const float4& cs, const float4& sn, const float* wv,
                                             int kk, float* dn) {
    const float cc[4] = {cs.x, cs.y, cs.z, cs.w}, ss[4] = {sn.x, sn.y, sn.z, sn.w};
    const float4 w0 = *reinterpret_cast<const float4*>(wv + kk), w1 = *reinterpret_cast<const float4*>(wv + kk + 4);
    const float ww[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const uint32_t g2 = word_of(gw, e);
        const float g0 = bf16_lo(g2), g1 = bf16_hi(g2);
        dn[2 * e] = __fmul_rn(__fadd_rn(__fmul_rn(g0, cc[e]), __fmul_rn(g1, ss[e])), ww[2 * e]);
        dn[2 * e + 1] = __fmul_rn(__fsub_rn(__fmul_rn(g1, cc[e]), __fmul_rn(g0, ss[e])), ww[2 * e + 1]);
    }
}

__global__ void __launch_bounds__(kQThreads, 1) quantize_norm_rope_kernel(const __grid_constant__ NormRopeArgs A) {
    extern __shared__ uint8_t smem_raw[];
    NormRopeSmem& sm = *reinterpret_cast<NormRopeSmem*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const QuantArgs& p = A.q;
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    uint32_t* const err = p.err;

    if (tid == 0) {
        for (int s = 0; s < kQStages; ++s) {
            mbar_init(smem_addr(&sm.full[s]), 1);
            mbar_init(smem_addr(&sm.empty[s]), kQConsumerWarps);
        }
        sm.abort = 0;
        fence_barrier_init();
    }
    if (tid < 2 * kNormRopeD) sm.w[tid / kNormRopeD][tid % kNormRopeD] =
        __ldg((tid < kNormRopeD ? A.wq : A.wk) + (tid % kNormRopeD));
    __syncthreads();
    grid_launch_dependents();
    grid_wait_prerequisites();

    if (warp == kQConsumerWarps) {
        if (lane_id() == 0) {
            prefetch_tensormap(&A.gmap);
            prefetch_tensormap(&A.xmap);
            int it = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < A.units && ok; u += gridDim.x) {
                const int tm = u / A.units_per_row, tk0 = (u % A.units_per_row) * A.span;
                const int tk1 = min(tk0 + A.span, p.tiles_k);
                for (int tk = tk0; tk < tk1; ++tk, ++it) {
                    const int s = it % kQStages;
                    const uint32_t ph = (it / kQStages) & 1;
                    if (!mbar_wait(smem_addr(&sm.empty[s]), ph ^ 1, err, kErrQuantProducer, &sm.abort)) {
                        ok = false;
                        break;
                    }
                    const bool qk = (tk % 3) != 2;
                    const uint32_t bar = smem_addr(&sm.full[s]);
                    mbar_arrive_expect_tx(bar, qk ? 2 * kQTileBytes : kQTileBytes);
                    tma_load_2d(smem_addr(sm.tile[s]), &A.gmap, tk * kQT, tm * kQT, bar);
                    tma_load_2d(smem_addr(sm.tile[s]) + kQBoxBytes, &A.gmap, tk * kQT + 64, tm * kQT, bar);
                    if (qk) {
                        tma_load_2d(smem_addr(sm.xt[s]), &A.xmap, tk * kQT, tm * kQT, bar);
                        tma_load_2d(smem_addr(sm.xt[s]) + kQBoxBytes, &A.xmap, tk * kQT + 64, tm * kQT, bar);
                    }
                }
            }
            const int armed = it < kQStages ? it : kQStages;
            for (int i = 1; i <= armed; ++i) {
                const int j = it - i;
                mbar_wait_quiet(smem_addr(&sm.full[j % kQStages]), (j / kQStages) & 1, kWaitLimitNs);
            }
        }
        return;
    }

    const uint32_t lane = lane_id();
    // the rowwise thread mapping of the quantizer: the two lanes that differ in bit 2 share a
    // row, each with two 32-column blocks b
    const int L = 4 * warp + (lane & 3);
    const int Q = lane >> 3;
    const int r = Q * 32 + L;
    int it = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < A.units && ok; u += gridDim.x) {
        const int tm = u / A.units_per_row, tk0 = (u % A.units_per_row) * A.span;
        const int tk1 = min(tk0 + A.span, p.tiles_k);
        const int64_t m0 = static_cast<int64_t>(tm) * kQT;
        const int64_t row = m0 + r;
        const bool live = row < p.M;
        const int64_t rrow = live ? row : 0;
        // this thread's RoPE cosines and sines for the unit: pairs 16 b .. 16 b + 15 of its row
        float4 cs4[2][4], sn4[2][4];
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int b = ((lane >> 2) & 1) + 2 * i;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                cs4[i][c] = __ldg(reinterpret_cast<const float4*>(A.cosv + rrow * 64) + 4 * b + c);
                sn4[i][c] = __ldg(reinterpret_cast<const float4*>(A.sinv + rrow * 64) + 4 * b + c);
            }
        }
        // and the row's saved r of every (head, part) of the unit, into shared memory: the two
        // lanes of the row split the loads, so each tile reads its value without a global load
        const int h0 = tk0 / 3, nh = (tk1 - 1) / 3 - h0 + 1;
        for (int k = static_cast<int>((lane >> 2) & 1); k < 2 * nh; k += 2)
            sm.rs[r][k] = live ? __ldg(A.rstd + (rrow * A.H + h0) * 2 + k) : 0.0f;
        __syncwarp();
        for (int tk = tk0; tk < tk1; ++tk, ++it) {
            const int s = it % kQStages;
            const uint32_t ph = (it / kQStages) & 1;
            int okw = 0;
            if (lane == 0) okw = mbar_wait(smem_addr(&sm.full[s]), ph, err, kErrQuantConsumer, &sm.abort) ? 1 : 0;
            // Every consumer warp meets every tile's barrier, with its ok flag: a warp whose
            // wait ran out skips the tile's work and all leave together.
            const bool have = __shfl_sync(0xFFFFFFFFu, okw, 0) != 0;
            const int part = tk % 3, head = tk / 3;
            const int64_t k0 = static_cast<int64_t>(tk) * kQT;
            const uint32_t tile = smem_addr(sm.tile[s]);
            const uint32_t xtile = smem_addr(sm.xt[s]);
            uint8_t* const atom_row = p.s_row + (static_cast<int64_t>(tm) * (p.kb_row >> 2) + tk) * 512;
            uint8_t* const atom_col = p.s_col + (static_cast<int64_t>(tk) * (p.kb_col >> 2) + tm) * 512;

            if (have && part != 2) {
                const float* const wv = sm.w[part];
                const float rr = sm.rs[r][(head - tk0 / 3) * 2 + part];
                float dot = 0.0f;
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int b = ((lane >> 2) & 1) + 2 * i;
                    const uint32_t box = tile + (b >> 1) * kQBoxBytes;
                    const uint32_t xbox = xtile + (b >> 1) * kQBoxBytes;
                    const int j0 = (b & 1) * 4;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const uint4 xw = lds128(xbox + swz(r, j0 + c));
                        float dn[8];
                        norm_rope_dn(lds128(box + swz(r, j0 + c)), cs4[i][c], sn4[i][c], wv, 32 * b + 8 * c, dn);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            dot = __fmaf_rn(dn[2 * e], bf16_lo(word_of(xw, e)), dot);
                            dot = __fmaf_rn(dn[2 * e + 1], bf16_hi(word_of(xw, e)), dot);
                        }
                    }
                }
                dot = __fadd_rn(dot, __shfl_xor_sync(0xFFFFFFFFu, dot, 4));
                const float coef = __fmul_rn(__fmul_rn(__fmul_rn(rr, rr), rr), __fmul_rn(dot, 1.0f / kNormRopeD));
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int b = ((lane >> 2) & 1) + 2 * i;
                    const uint32_t box = tile + (b >> 1) * kQBoxBytes;
                    const uint32_t xbox = xtile + (b >> 1) * kQBoxBytes;
                    const int j0 = (b & 1) * 4;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const uint4 xw = lds128(xbox + swz(r, j0 + c));
                        float dn[8];
                        norm_rope_dn(lds128(box + swz(r, j0 + c)), cs4[i][c], sn4[i][c], wv, 32 * b + 8 * c, dn);
                        uint32_t o[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const uint32_t xwd = word_of(xw, e);
                            const float d0 = __fsub_rn(__fmul_rn(rr, dn[2 * e]), __fmul_rn(coef, bf16_lo(xwd)));
                            const float d1 = __fsub_rn(__fmul_rn(rr, dn[2 * e + 1]), __fmul_rn(coef, bf16_hi(xwd)));
                            __nv_bfloat162 h2 = __floats2bfloat162_rn(d0, d1);
                            // rows past M stay +0 padding (a zero gradient can still give -0)
                            o[e] = live ? *reinterpret_cast<uint32_t*>(&h2) : 0u;
                        }
                        sts128q(box + swz(r, j0 + c), make_uint4(o[0], o[1], o[2], o[3]));
                    }
                }
            }
            if (have) {
                uint4 v[2][4];
        #pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int b = ((lane >> 2) & 1) + 2 * i;
                    const uint32_t box = tile + (b >> 1) * kQBoxBytes;
                    const int j0 = (b & 1) * 4;
        #pragma unroll
                    for (int c = 0; c < 4; ++c) v[i][c] = lds128(box + swz(r, j0 + c));
                }
                if (A.dmixed != nullptr && row < p.M) {
        #pragma unroll
                    for (int i = 0; i < 2; ++i) {
                        const int b = ((lane >> 2) & 1) + 2 * i;
        #pragma unroll
                        for (int c = 0; c < 4; ++c)
                            *reinterpret_cast<uint4*>(A.dmixed + row * p.K + k0 + 32 * b + 8 * c) = v[i][c];
                    }
                }
        #pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const int b = ((lane >> 2) & 1) + 2 * i;
                    uint32_t m = absmax2(absmax2(absmax2(v[i][0].x, v[i][0].y), absmax2(v[i][0].z, v[i][0].w)),
                                         absmax2(absmax2(v[i][1].x, v[i][1].y), absmax2(v[i][1].z, v[i][1].w)));
                    m = absmax2(m, absmax2(absmax2(absmax2(v[i][2].x, v[i][2].y), absmax2(v[i][2].z, v[i][2].w)),
                                           absmax2(absmax2(v[i][3].x, v[i][3].y), absmax2(v[i][3].z, v[i][3].w))));
                    m = absmax2(m, m >> 16) & 0x7FFFu;
                    const uint32_t byte = scale_byte(m);
                    const uint32_t inv = inv_scale_bits(byte);
                    const uint64_t s2 = pack2(inv, inv);
                    const uint4 q = make_uint4(encode8(v[i][0].x, v[i][0].y, v[i][0].z, v[i][0].w, s2),
                                               encode8(v[i][1].x, v[i][1].y, v[i][1].z, v[i][1].w, s2),
                                               encode8(v[i][2].x, v[i][2].y, v[i][2].z, v[i][2].w, s2),
                                               encode8(v[i][3].x, v[i][3].y, v[i][3].z, v[i][3].w, s2));
                    if (row < p.M) {
                        *reinterpret_cast<uint4*>(p.q_row + row * p.ldq_row + ((k0 + 32 * b) >> 1)) = q;
                        if (!p.tc_layout) p.s_row[row * p.kb_row + (k0 >> 5) + b] = static_cast<uint8_t>(byte);
                    }
                    if (p.tc_layout) atom_row[L * 16 + Q * 4 + b] = static_cast<uint8_t>(row < p.M ? byte : 0u);
                }
                // every warp's rows of dx are in the stage before any column is read
            }
            if (!named_barrier_and(kBarConsumers, kQConsumers, have)) {
                ok = false;
                break;
            }

            // ---- columnwise, as the quantizer's plain columnwise pass
            {
                const int pc = 8 * warp + (lane & 7), rb = lane >> 3;
                const uint32_t box = tile + (pc >> 5) * kQBoxBytes;
                const int jc = (pc & 31) >> 2;
                const uint32_t inner = (pc & 3) * 4;
                uint32_t toff[8];
    #pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int rr2 = k ^ (2 * rb);
                    toff[k] = box + rb * 32 * 128 + rr2 * 128 + ((jc ^ rr2) << 4) + inner;
                }
                uint32_t w[32];
    #pragma unroll
                for (int i = 0; i < 32; ++i) w[i] = lds32(toff[i & 7] + (i & ~7) * 128);
                const uint32_t sel = 0x3210u ^ (0x1111u * static_cast<uint32_t>(rb));
                const int64_t kc = k0 + 2 * pc;
                uint32_t m = w[0];
    #pragma unroll
                for (int i = 1; i < 32; ++i) m = absmax2(m, w[i]);
                const uint32_t byte0 = scale_byte(m), byte1 = scale_byte(m >> 16);
                const uint64_t s2 = pack2(inv_scale_bits(byte0), inv_scale_bits(byte1));
                uint32_t q0[4], q1[4];
    #pragma unroll
                for (int j = 0; j < 4; ++j) {
                    encode_cols8(&w[8 * j], s2, &q0[j], &q1[j]);
                    q0[j] = __byte_perm(q0[j], 0, sel);
                    q1[j] = __byte_perm(q1[j], 0, sel);
                }
                const int64_t off = (m0 + rb * 32) >> 1;
                if (kc < p.K) {
                    *reinterpret_cast<uint4*>(p.q_col + kc * p.ldq_col + off) = make_uint4(q0[0], q0[1], q0[2], q0[3]);
                    if (!p.tc_layout) p.s_col[kc * p.kb_col + (m0 >> 5) + rb] = static_cast<uint8_t>(byte0);
                }
                if (kc + 1 < p.K) {
                    *reinterpret_cast<uint4*>(p.q_col + (kc + 1) * p.ldq_col + off) = make_uint4(q1[0], q1[1], q1[2], q1[3]);
                    if (!p.tc_layout) p.s_col[(kc + 1) * p.kb_col + (m0 >> 5) + rb] = static_cast<uint8_t>(byte1);
                }
                const int kl0 = 2 * pc, kl1 = 2 * pc + 1;
                if (p.tc_layout) {
                    atom_col[(kl0 & 31) * 16 + (kl0 >> 5) * 4 + rb] = static_cast<uint8_t>(kc < p.K ? byte0 : 0u);
                    atom_col[(kl1 & 31) * 16 + (kl1 >> 5) * 4 + rb] = static_cast<uint8_t>(kc + 1 < p.K ? byte1 : 0u);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&sm.empty[s]));
        }
    }
}

}  // namespace

size_t quantize_smem_bytes() { return sizeof(QuantSmem) + 1024; }
int quantize_ctas_per_sm(bool sr) { return sr ? 1 : kQCtasPerSm; }

size_t quantize_norm_rope_smem_bytes() { return sizeof(NormRopeSmem) + 1024; }
int quantize_norm_rope_ctas_per_sm() { return 1; }

cudaError_t launch_quantize_norm_rope(const NormRopeArgs& a, int grid, cudaStream_t stream) {
    const size_t smem = quantize_norm_rope_smem_bytes();
    cudaError_t e = cudaFuncSetAttribute(quantize_norm_rope_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kQThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, quantize_norm_rope_kernel, a);
}

__global__ void amax_zero_kernel(const __grid_constant__ QuantBatch B) {
    if (static_cast<int>(threadIdx.x) < B.count && B.args[threadIdx.x].amax_bits != nullptr)
        *B.args[threadIdx.x].amax_bits = 0u;
}

cudaError_t launch_quantize(const QuantBatch& b, bool dual, bool sr, int grid, cudaStream_t stream) {
    const size_t smem = quantize_smem_bytes();
    bool any_amax = false;
    for (int j = 0; j < b.count; ++j) any_amax = any_amax || b.args[j].amax_bits != nullptr;
    if (any_amax) {   // a plain launch: the quantizer's dependency wait covers it
        amax_zero_kernel<<<1, 32, 0, stream>>>(b);
        const cudaError_t ez = cudaGetLastError();
        if (ez != cudaSuccess) return ez;
    }
    if (sr && !dual) return cudaErrorInvalidValue;
    bool recipes = false, any_2d = false;
    for (int j = 0; j < b.count; ++j) {
        recipes = recipes || b.args[j].block_2d != 0 || b.args[j].rht != 0;
        any_2d = any_2d || b.args[j].block_2d != 0;
    }
    if (sr && any_2d) return cudaErrorInvalidValue;   // 2-D blocks are a weight recipe, without SR
    auto k = sr        ? (recipes ? quantize_kernel<true, true, true> : quantize_kernel<true, true, false>)
             : recipes ? (dual ? quantize_kernel<true, false, true> : quantize_kernel<false, false, true>)
                       : (dual ? quantize_kernel<true, false, false> : quantize_kernel<false, false, false>);
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kQThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, b);
}

}  // namespace mxfp4
