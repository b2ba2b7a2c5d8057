/*
 * mxfp4_oracle.c -- plain, slow CPU oracle for MXFP4 block-scaled quantization and the
 * block-scaled GEMM that consumes it.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or load this
 * file: only the tests, the package's smoke check and the CPU-baseline leg of the
 * benchmark use it.  It shares no code, header, table or constant with the CUDA
 * library.
 *
 * What it computes, and the passages it follows:
 *
 *  - Element and scale formats: FP4 E2M1 elements packed two per byte
 *    (torch.float4_e2m1fn_x2) and one E8M0 scale byte per block (torch.float8_e8m0fnu),
 *    as the output dtypes of `_quantize_mxfp4_dual_fake` in primus_turbo_mxfp4_local.py
 *    declare them.
 *  - Block size 32 (MXFP4_BLOCK_SIZE) and padding of the packed dimension to a multiple
 *    of 128 (MXFP4_PADDING_ALIGN_SIZE), primus_turbo_mxfp4_local.py, module constants and
 *    the M_pad / N_pad arithmetic of `_quantize_mxfp4_dual_fake`.
 *  - Row blob of X[R,K]: q[R, Kp/2], s[R, Kp/32]; col blob: the row blob of X^T
 *    (same function, non-shuffled branch).
 *  - The GEMM C = A . B^T over K-packed operands, the form the forward, dgrad and wgrad
 *    calls of `MXFP4LinearFunction` in primus_turbo_mxfp4_local.py all take.
 *
 * The pages print no formula for the quantization itself.  The oracle follows the OCP
 * Microscaling (MX) v1.0 rule for MXFP4:
 *   scale exponent e = floor(log2(amax)) - 2   (2 = the largest E2M1 exponent),
 *   clamped to the E8M0 range [-127, 127]; an all-zero block gets the byte 0x00;
 *   element = round-to-nearest-even of v / 2^e onto {0, 0.5, 1, 1.5, 2, 3, 4, 6},
 *   saturating at 6.
 * Readings taken where that rule is silent:
 *   - the sign of an element that rounds to zero is kept (-0 encodes as 0x8);
 *   - padding elements are +0, so an all-padding block gets the byte 0x00;
 *   - the low nibble of byte j holds element 2j, the high nibble element 2j+1;
 *   - inputs must be finite; the quantizers return -1 on a NaN or infinity.
 *
 * Everything is computed in fp64, where every step above is exact.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define BLOCK 32
#define PAD 128

static int64_t cdiv64(int64_t a, int64_t b) { return (a + b - 1) / b; }

/* bf16 bit pattern -> double (exact: bf16 is the top half of an IEEE binary32). */
double oracle_bf16_to_f64(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* E2M1 code (bit 3 sign, bits 2..1 exponent with bias 1, bit 0 mantissa) -> value. */
double oracle_e2m1_decode(uint8_t code) {
    int sign = (code >> 3) & 1;
    int exp = (code >> 1) & 3;
    int man = code & 1;
    double mag = (exp == 0) ? 0.5 * man                       /* subnormal: 0 or 0.5 */
                            : ldexp(1.0 + 0.5 * man, exp - 1); /* 1, 1.5, 2, 3, 4, 6 */
    return sign ? -mag : mag;
}

/* Finite double -> E2M1 code: IEEE round-to-nearest-even onto the E2M1 grid, then
 * saturation of anything above 6 to 6.  Within a binade the representable magnitudes
 * are consecutive multiples of a quantum (0.5 below 2, 1 in [2,4), 2 in [4,8)), and an
 * even multiple is an even code, so rounding v/quantum half-to-even rounds ties to the
 * even code.  The sign bit is the sign of v, also when the magnitude rounds to 0. */
uint8_t oracle_e2m1_encode(double v) {
    uint8_t sign = signbit(v) ? 0x8 : 0x0;
    double a = fabs(v);
    double quantum = (a < 2.0) ? 0.5 : (a < 4.0) ? 1.0 : 2.0;
    double r = nearbyint(a / quantum) * quantum; /* default rounding mode: ties-to-even */
    if (r > 6.0) r = 6.0;
    uint8_t mag;
    if (r == 0.0) mag = 0;
    else if (r == 0.5) mag = 1;
    else if (r == 1.0) mag = 2;
    else if (r == 1.5) mag = 3;
    else if (r == 2.0) mag = 4;
    else if (r == 3.0) mag = 5;
    else if (r == 4.0) mag = 6;
    else mag = 7; /* 6.0 */
    return sign | mag;
}

/* Shared scale of a block whose largest magnitude is amax (finite, >= 0), as the E8M0
 * byte (unbiased exponent + 127).  floor(log2(amax)) comes from frexp: amax = f * 2^E
 * with f in [0.5, 1), so floor(log2(amax)) = E - 1. */
uint8_t oracle_e8m0_scale(double amax) {
    if (amax == 0.0) return 0;
    int E;
    frexp(amax, &E);
    int e = (E - 1) - 2;
    if (e < -127) e = -127;
    if (e > 127) e = 127;
    return (uint8_t)(e + 127);
}

/* Quantize one block of 32 values (padding already +0): writes 16 packed bytes and the
 * scale byte.  Returns -1 if a value is not finite. */
static int quantize_block(const double v[BLOCK], uint8_t q[BLOCK / 2], uint8_t* s) {
    double amax = 0.0;
    for (int i = 0; i < BLOCK; ++i) {
        if (!isfinite(v[i])) return -1;
        if (fabs(v[i]) > amax) amax = fabs(v[i]);
    }
    uint8_t byte = oracle_e8m0_scale(amax);
    int e = (int)byte - 127;
    for (int j = 0; j < BLOCK / 2; ++j) {
        uint8_t lo = oracle_e2m1_encode(ldexp(v[2 * j], -e));
        uint8_t hi = oracle_e2m1_encode(ldexp(v[2 * j + 1], -e));
        q[j] = (uint8_t)(lo | (hi << 4));
    }
    *s = byte;
    return 0;
}

/* Row blob of X[M,K] (bf16 bits, row pitch ldx elements): blocks of 32 run along K.
 * q: [M, Kp/2] bytes, s: [M, Kp/32] bytes (plain layout).  Kp = ceil(K/128)*128. */
int oracle_quantize_row(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, uint8_t* q,
                        uint8_t* s) {
    int64_t Kp = cdiv64(K, PAD) * PAD, KB = Kp / BLOCK;
    double v[BLOCK];
    for (int64_t r = 0; r < M; ++r) {
        for (int64_t b = 0; b < KB; ++b) {
            for (int i = 0; i < BLOCK; ++i) {
                int64_t k = b * BLOCK + i;
                v[i] = (k < K) ? oracle_bf16_to_f64(x[r * ldx + k]) : 0.0;
            }
            if (quantize_block(v, q + r * (Kp / 2) + b * (BLOCK / 2), s + r * KB + b)) return -1;
        }
    }
    return 0;
}

/* Col blob of X[M,K]: the row blob of X^T, i.e. blocks of 32 run along M.
 * q: [K, Mp/2] bytes, s: [K, Mp/32] bytes (plain layout).  Mp = ceil(M/128)*128. */
int oracle_quantize_col(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, uint8_t* q,
                        uint8_t* s) {
    int64_t Mp = cdiv64(M, PAD) * PAD, MB = Mp / BLOCK;
    double v[BLOCK];
    for (int64_t k = 0; k < K; ++k) {
        for (int64_t b = 0; b < MB; ++b) {
            for (int i = 0; i < BLOCK; ++i) {
                int64_t m = b * BLOCK + i;
                v[i] = (m < M) ? oracle_bf16_to_f64(x[m * ldx + k]) : 0.0;
            }
            if (quantize_block(v, q + k * (Mp / 2) + b * (BLOCK / 2), s + k * MB + b)) return -1;
        }
    }
    return 0;
}

/* Scale bytes of a blob with R rows and KB (a multiple of 4) blocks per row, from the
 * plain layout s[R, KB] into the tensor-core layout: rows padded to a multiple of 128 and
 * tiled in 128-row x 4-block atoms of 512 bytes, atoms ordered block-group-fastest; inside
 * an atom, byte (r, kb) sits at (r % 32) * 16 + (r / 32) * 4 + kb, i.e. 32 lines of 16
 * bytes.  Padding rows hold 0x00.  out must hold ceil(R/128)*128*KB bytes. */
void oracle_scale_to_tc(const uint8_t* s, int64_t R, int64_t KB, uint8_t* out) {
    int64_t Rp = cdiv64(R, PAD) * PAD;
    memset(out, 0, (size_t)(Rp * KB));
    for (int64_t r = 0; r < R; ++r)
        for (int64_t kb = 0; kb < KB; ++kb) {
            int64_t atom = (r / 128) * (KB / 4) + kb / 4;
            int64_t within = (r % 32) * 16 + ((r % 128) / 32) * 4 + (kb % 4);
            out[atom * 512 + within] = s[r * KB + kb];
        }
}

/* Dequantize a blob (plain scale layout) with R rows and Kp (multiple of 128) packed
 * elements per row into out[R, Kp]: value = E2M1(code) * 2^(scale - 127). */
void oracle_dequantize(const uint8_t* q, const uint8_t* s, int64_t R, int64_t Kp, double* out) {
    int64_t KB = Kp / BLOCK;
    for (int64_t r = 0; r < R; ++r)
        for (int64_t k = 0; k < Kp; ++k) {
            uint8_t byte = q[r * (Kp / 2) + k / 2];
            uint8_t code = (k & 1) ? (byte >> 4) : (byte & 0xF);
            out[r * Kp + k] = ldexp(oracle_e2m1_decode(code), (int)s[r * KB + k / BLOCK] - 127);
        }
}

/* C[m,n] = sum_{k<Kp} A[m,k] * B[n,k] in fp64 over dequantized rows A[M,Kp], B[N,Kp]
 * (both K-packed, the "TN" form), and cabs[m,n] = sum_k |A[m,k] * B[n,k]|, the scale the
 * accuracy bound is stated against.  Either output may be NULL.  Only rows
 * m in [m0, m1) of C are computed; c / cabs are indexed [m - m0, n]. */
void oracle_gemm_f64(const double* a, const double* b, int64_t M, int64_t N, int64_t Kp,
                     int64_t m0, int64_t m1, double* c, double* cabs) {
    (void)M;
    for (int64_t m = m0; m < m1; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0, accabs = 0.0;
            for (int64_t k = 0; k < Kp; ++k) {
                double p = a[m * Kp + k] * b[n * Kp + k];
                acc += p;
                accabs += fabs(p);
            }
            if (c) c[(m - m0) * N + n] = acc;
            if (cabs) cabs[(m - m0) * N + n] = accabs;
        }
}

/* Round finite doubles to bf16 bit patterns, round-to-nearest-even, once.  bf16 keeps 8
 * significant bits and the binary32 exponent range (normal down to 2^-126, subnormal
 * spacing 2^-133); results beyond the largest finite value become infinity. */
void oracle_round_to_bf16(const double* in, uint16_t* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) {
        double x = in[i];
        uint16_t sign = signbit(x) ? 0x8000 : 0;
        double a = fabs(x);
        if (a == 0.0) { out[i] = sign; continue; }
        int E;
        frexp(a, &E); /* a in [2^(E-1), 2^E) */
        int e = E - 1;
        double quantum = (e < -126) ? ldexp(1.0, -133) : ldexp(1.0, e - 7);
        double r = nearbyint(a / quantum) * quantum;
        if (r >= ldexp(1.0, 128)) { out[i] = sign | 0x7F80; continue; }
        float f = (float)r; /* exact: r has at most 8 significant bits in bf16 range */
        uint32_t u;
        memcpy(&u, &f, sizeof u);
        out[i] = sign | (uint16_t)(u >> 16);
    }
}

/* The layer's bias add after the GEMM: `output + bias` in `_forward_impl` of
 * MXFP4ColumnParallelLinear / MXFP4RowParallelLinear (primus_turbo_mxfp4_local.py), where
 * `output` is the GEMM result already in the output dtype and `bias` a bf16 vector added
 * to every row.  Computed the way an elementwise add of those dtypes is defined: both
 * operands widened exactly to binary32, one binary32 addition (round to nearest even),
 * and for a bf16 result one more round-to-nearest-even to bf16.  y and out are [M, N]
 * row-major; bias is [N]. */
static float bf16_bits_to_f32(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

void oracle_bias_add_bf16(const uint16_t* y, const uint16_t* bias, int64_t M, int64_t N, uint16_t* out) {
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            volatile float s = bf16_bits_to_f32(y[m * N + n]) + bf16_bits_to_f32(bias[n]);
            double d = (double)s;
            oracle_round_to_bf16(&d, &out[m * N + n], 1);
        }
}

void oracle_bias_add_f32(const float* y, const uint16_t* bias, int64_t M, int64_t N, float* out) {
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            volatile float s = y[m * N + n] + bf16_bits_to_f32(bias[n]);
            out[m * N + n] = s;
        }
}

/* ---------------------------------------------------------------------------------------
 * Stochastic rounding of the elements (the `rowwise_use_sr` / `colwise_use_sr` flags that
 * `_quantize_grad_dual` in primus_turbo_mxfp4_local.py sets from `use_sr`, i.e. from the
 * layer's `mxfp4_gradient_stochastic_rounding` option; the pages name the flag and apply
 * it to gradients only, and define nothing more).  Reading taken:
 *   - the scale byte is the one of the round-to-nearest quantizer (the flag names the
 *     element rounding only);
 *   - a scaled element y with |y| >= 6 becomes 6 (saturation, as without the flag);
 *     otherwise, with lo <= |y| < hi its two neighbours on {0, .5, 1, 1.5, 2, 3, 4, 6} and
 *     P = (|y| - lo) / (hi - lo), the magnitude is hi when r < floor(P * 2^16) and lo
 *     otherwise, r being 16 random bits of the element; the sign is kept;
 *   - the random bits come from Philox4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel
 *     random numbers: as easy as 1, 2, 3", SC 2011), key = (seed low word, seed high
 *     word), counter = (b / 8, a, packing, 0) for the element in row a, column b of the
 *     blob being packed (packing 0: row blob of X; 1: col blob, i.e. row a = column of X,
 *     b = row of X); of the four output words, word (b / 2) % 4 holds the element's bits
 *     in its low half when b is even, its high half when b is odd.
 * -------------------------------------------------------------------------------------- */

/* One Philox4x32 round: two 32x32 -> 64-bit products, then the published permutation
 * and key mixing. */
static void philox_round(uint32_t c[4], const uint32_t k[2]) {
    uint64_t p0 = (uint64_t)0xD2511F53u * c[0];
    uint64_t p1 = (uint64_t)0xCD9E8D57u * c[2];
    uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
    uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
    uint32_t n0 = hi1 ^ c[1] ^ k[0];
    uint32_t n2 = hi0 ^ c[3] ^ k[1];
    c[0] = n0;
    c[1] = lo1;
    c[2] = n2;
    c[3] = lo0;
}

/* Philox4x32 with 10 rounds; the key is bumped by the Weyl constants between rounds. */
void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
    uint32_t c[4] = {ctr[0], ctr[1], ctr[2], ctr[3]};
    uint32_t k[2] = {key[0], key[1]};
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k[0] += 0x9E3779B9u;
            k[1] += 0xBB67AE85u;
        }
        philox_round(c, k);
    }
    for (int i = 0; i < 4; ++i) out[i] = c[i];
}

/* The 16 random bits of blob element (row a, column b) in the given packing. */
uint32_t oracle_sr_bits(uint64_t seed, int64_t a, int64_t b, int packing) {
    uint32_t ctr[4] = {(uint32_t)(b / 8), (uint32_t)a, (uint32_t)packing, 0u};
    uint32_t key[2] = {(uint32_t)(seed & 0xFFFFFFFFu), (uint32_t)(seed >> 32)};
    uint32_t w[4];
    oracle_philox4x32_10(ctr, key, w);
    uint32_t word = w[(b / 2) % 4];
    return (b % 2) ? (word >> 16) : (word & 0xFFFFu);
}

/* E2M1 code of the scaled element y under stochastic rounding with 16 random bits r. */
uint8_t oracle_e2m1_encode_sr(double y, uint32_t r) {
    static const double grid[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
    uint8_t sign = signbit(y) ? 0x8 : 0x0;
    double a = fabs(y);
    if (a >= 6.0) return sign | 7;
    int lo = 0;
    while (grid[lo + 1] <= a) ++lo; /* grid[lo] <= a < grid[lo + 1] */
    double p = (a - grid[lo]) / (grid[lo + 1] - grid[lo]); /* exact: the gap is 2^-1, 2^0 or 2^1 */
    double t = floor(p * 65536.0);
    return sign | (uint8_t)(((double)r < t) ? lo + 1 : lo);
}

static int quantize_block_sr(const double v[BLOCK], uint8_t q[BLOCK / 2], uint8_t* s, uint64_t seed,
                             int64_t a, int64_t b0, int packing) {
    double amax = 0.0;
    for (int i = 0; i < BLOCK; ++i) {
        if (!isfinite(v[i])) return -1;
        if (fabs(v[i]) > amax) amax = fabs(v[i]);
    }
    uint8_t byte = oracle_e8m0_scale(amax);
    int e = (int)byte - 127;
    for (int j = 0; j < BLOCK / 2; ++j) {
        uint8_t lo = oracle_e2m1_encode_sr(ldexp(v[2 * j], -e), oracle_sr_bits(seed, a, b0 + 2 * j, packing));
        uint8_t hi = oracle_e2m1_encode_sr(ldexp(v[2 * j + 1], -e), oracle_sr_bits(seed, a, b0 + 2 * j + 1, packing));
        q[j] = (uint8_t)(lo | (hi << 4));
    }
    *s = byte;
    return 0;
}

/* Row blob of X[M,K] with stochastic rounding (packing 0); layout as oracle_quantize_row.
 * row_ids (may be NULL): the row index a of each of the M rows in the full tensor, for
 * quantizing sampled rows with the random bits of their true position. */
int oracle_quantize_row_sr(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, uint8_t* q, uint8_t* s,
                           uint64_t seed, const int64_t* row_ids) {
    int64_t Kp = cdiv64(K, PAD) * PAD, KB = Kp / BLOCK;
    double v[BLOCK];
    for (int64_t r = 0; r < M; ++r)
        for (int64_t b = 0; b < KB; ++b) {
            for (int i = 0; i < BLOCK; ++i) {
                int64_t k = b * BLOCK + i;
                v[i] = (k < K) ? oracle_bf16_to_f64(x[r * ldx + k]) : 0.0;
            }
            if (quantize_block_sr(v, q + r * (Kp / 2) + b * (BLOCK / 2), s + r * KB + b, seed,
                                  row_ids ? row_ids[r] : r, b * BLOCK, 0))
                return -1;
        }
    return 0;
}

/* Col blob of X[M,K] with stochastic rounding (packing 1): the row blob of X^T, its row a
 * being column a of X; layout as oracle_quantize_col.  col_ids (may be NULL): the column
 * index of each of the K columns in the full tensor. */
int oracle_quantize_col_sr(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, uint8_t* q, uint8_t* s,
                           uint64_t seed, const int64_t* col_ids) {
    int64_t Mp = cdiv64(M, PAD) * PAD, MB = Mp / BLOCK;
    double v[BLOCK];
    for (int64_t k = 0; k < K; ++k)
        for (int64_t b = 0; b < MB; ++b) {
            for (int i = 0; i < BLOCK; ++i) {
                int64_t m = b * BLOCK + i;
                v[i] = (m < M) ? oracle_bf16_to_f64(x[m * ldx + k]) : 0.0;
            }
            if (quantize_block_sr(v, q + k * (Mp / 2) + b * (BLOCK / 2), s + k * MB + b, seed,
                                  col_ids ? col_ids[k] : k, b * BLOCK, 1))
                return -1;
        }
    return 0;
}

/* ---------------------------------------------------------------------------------------
 * Hybrid FP8 backward (`backward_is_fp8` in `MXFP4LinearFunction.backward`,
 * primus_turbo_mxfp4_local.py): dY, X and W are quantized tensorwise to FP8 E5M2
 * (`_quantize_fp8_tw(…, fp8_bwd_dtype)`, the dtype being `float8_e5m2` and the granularity
 * TENSORWISE in the parallel-linear constructors) and dgrad / wgrad run as FP8 GEMMs
 * (`gemm_fp8_impl`) whose result carries the two tensors' inverse scales.  The pages call
 * `_quantize_fp8_tw` without defining it; reading taken (the usual tensorwise recipe):
 *   amax = max |x| over the tensor; scale = 57344 / amax in binary32 (57344 = the largest
 *   finite E5M2 value), the largest finite binary32 if that overflows, 1 if amax = 0;
 *   element = E5M2 round-to-nearest-even of (binary32) x * scale, saturating at +-57344,
 *   sign of zero kept; scale_inv = 1 / scale in binary32.
 * GEMM: C = (sum_k a_k b_k) * s with s = a_scale_inv * b_scale_inv rounded to binary32.
 * -------------------------------------------------------------------------------------- */

/* E5M2 code (bit 7 sign, bits 6..2 exponent with bias 15, bits 1..0 mantissa) -> value. */
double oracle_e5m2_decode(uint8_t code) {
    int sign = (code >> 7) & 1;
    int exp = (code >> 2) & 31;
    int man = code & 3;
    double mag;
    if (exp == 0) mag = ldexp((double)man, -16);              /* subnormal: man * 2^-16 */
    else if (exp == 31) mag = man ? NAN : INFINITY;
    else mag = ldexp(1.0 + man / 4.0, exp - 15);
    return sign ? -mag : mag;
}

/* Round-to-nearest-even of a finite value onto E5M2, saturating at +-57344. */
uint8_t oracle_e5m2_encode(double v) {
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs(v);
    if (a >= 57344.0) return sign | 0x7B;                     /* 1.75 * 2^15 */
    double quantum;
    if (a < ldexp(1.0, -14)) {
        quantum = ldexp(1.0, -16);                             /* subnormal spacing */
    } else {
        int E;
        frexp(a, &E);                                          /* a in [2^(E-1), 2^E) */
        quantum = ldexp(1.0, (E - 1) - 2);                     /* 2 mantissa bits */
    }
    double r = nearbyint(a / quantum) * quantum;
    if (r >= 57344.0) return sign | 0x7B;
    if (r == 0.0) return sign;
    int E;
    frexp(r, &E);
    int e = E - 1;
    if (e < -14) return sign | (uint8_t)(r / ldexp(1.0, -16)); /* subnormal */
    int man = (int)((r / ldexp(1.0, e) - 1.0) * 4.0);
    return sign | (uint8_t)(((e + 15) << 2) | man);
}

/* Tensorwise E5M2 quantization of X[M,K] (bf16 bits, pitch ldx): q_row [M, ldr] holds X's
 * codes (may be NULL), q_col [K, ldc] the codes of X^T (may be NULL); pitches in bytes,
 * bytes past K (row copy) or M (col copy) are 0x00.  Writes amax and scale_inv.  Returns
 * -1 on a non-finite input. */
int oracle_fp8_quantize_tw(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, uint8_t* q_row, int64_t ldr,
                           uint8_t* q_col, int64_t ldc, float* amax_out, float* scale_inv_out) {
    float amax = 0.0f;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t k = 0; k < K; ++k) {
            float v = bf16_bits_to_f32(x[m * ldx + k]);
            if (!isfinite(v)) return -1;
            if (fabsf(v) > amax) amax = fabsf(v);
        }
    volatile float scale = 1.0f;
    if (amax > 0.0f) {
        scale = 57344.0f / amax;
        if (isinf(scale)) scale = FLT_MAX;
    }
    volatile float inv = 1.0f / scale;
    if (q_row) memset(q_row, 0, (size_t)(M * ldr));
    if (q_col) memset(q_col, 0, (size_t)(K * ldc));
    for (int64_t m = 0; m < M; ++m)
        for (int64_t k = 0; k < K; ++k) {
            volatile float y = bf16_bits_to_f32(x[m * ldx + k]) * scale;
            uint8_t c = oracle_e5m2_encode((double)y);
            if (q_row) q_row[m * ldr + k] = c;
            if (q_col) q_col[k * ldc + m] = c;
        }
    *amax_out = amax;
    *scale_inv_out = inv;
    return 0;
}

/* Codes [R, ld] (first Kc columns used) -> fp64 values [R, Kc]. */
void oracle_fp8_dequantize(const uint8_t* q, int64_t R, int64_t Kc, int64_t ld, double* out) {
    for (int64_t r = 0; r < R; ++r)
        for (int64_t k = 0; k < Kc; ++k) out[r * Kc + k] = oracle_e5m2_decode(q[r * ld + k]);
}

/* The GEMM's output scale: the two inverse scales multiplied in binary32. */
float oracle_fp8_output_scale(float a_scale_inv, float b_scale_inv) {
    volatile float s = a_scale_inv * b_scale_inv;
    return s;
}

/* ---------------------------------------------------------------------------------------
 * 2-D block scales for weights: `_quantize_weight_dual` in primus_turbo_mxfp4_local.py sets
 * `rowwise_use_2d_block` and `colwise_use_2d_block` for the weight (activations and
 * gradients keep 1 x 32 blocks).  The pages name the flags only; reading taken: W is cut
 * into 32 x 32 blocks (padding +0), each block gets one E8M0 scale from the amax of its
 * 1024 elements by the same rule as a 1 x 32 block, and every element of the block is
 * encoded with that scale in both packings.  So the row blob's scale of (row r, block kb)
 * and the col blob's scale of (column k, block mb) are the scale of the 2-D block that
 * holds them, and the two blobs dequantize to exact transposes of each other.
 * -------------------------------------------------------------------------------------- */

/* Scale bytes of the 2-D blocks of X[M,K]: s2d[ceil(M/32), Kp/32]. */
static int block2d_scales(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, uint8_t* s2d) {
    int64_t Kp = cdiv64(K, PAD) * PAD, KB = Kp / BLOCK, MB = cdiv64(M, BLOCK);
    for (int64_t mb = 0; mb < MB; ++mb)
        for (int64_t kb = 0; kb < KB; ++kb) {
            double amax = 0.0;
            for (int64_t i = 0; i < BLOCK; ++i)
                for (int64_t j = 0; j < BLOCK; ++j) {
                    int64_t m = mb * BLOCK + i, k = kb * BLOCK + j;
                    if (m >= M || k >= K) continue;
                    double v = oracle_bf16_to_f64(x[m * ldx + k]);
                    if (!isfinite(v)) return -1;
                    if (fabs(v) > amax) amax = fabs(v);
                }
            s2d[mb * KB + kb] = oracle_e8m0_scale(amax);
        }
    return 0;
}

/* Row blob of X[M,K] with 2-D block scales; layout as oracle_quantize_row. */
int oracle_quantize_row_2d(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, uint8_t* q, uint8_t* s) {
    int64_t Kp = cdiv64(K, PAD) * PAD, KB = Kp / BLOCK, MB = cdiv64(M, BLOCK);
    uint8_t* s2d = (uint8_t*)malloc((size_t)(MB * KB));
    if (!s2d) return -2;
    if (block2d_scales(x, M, K, ldx, s2d)) { free(s2d); return -1; }
    for (int64_t r = 0; r < M; ++r)
        for (int64_t kb = 0; kb < KB; ++kb) {
            uint8_t byte = s2d[(r / BLOCK) * KB + kb];
            int e = (int)byte - 127;
            for (int j = 0; j < BLOCK / 2; ++j) {
                int64_t k0 = kb * BLOCK + 2 * j, k1 = k0 + 1;
                double v0 = (k0 < K) ? oracle_bf16_to_f64(x[r * ldx + k0]) : 0.0;
                double v1 = (k1 < K) ? oracle_bf16_to_f64(x[r * ldx + k1]) : 0.0;
                uint8_t lo = oracle_e2m1_encode(ldexp(v0, -e));
                uint8_t hi = oracle_e2m1_encode(ldexp(v1, -e));
                q[r * (Kp / 2) + kb * (BLOCK / 2) + j] = (uint8_t)(lo | (hi << 4));
            }
            s[r * KB + kb] = byte;
        }
    free(s2d);
    return 0;
}

/* Col blob of X[M,K] with 2-D block scales: the row blob of X^T, the 2-D blocks being the
 * same; layout as oracle_quantize_col. */
int oracle_quantize_col_2d(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, uint8_t* q, uint8_t* s) {
    int64_t Kp = cdiv64(K, PAD) * PAD, KB = Kp / BLOCK;
    int64_t Mp = cdiv64(M, PAD) * PAD, MBp = Mp / BLOCK, MB = cdiv64(M, BLOCK);
    uint8_t* s2d = (uint8_t*)malloc((size_t)(MB * KB));
    if (!s2d) return -2;
    if (block2d_scales(x, M, K, ldx, s2d)) { free(s2d); return -1; }
    for (int64_t k = 0; k < K; ++k)
        for (int64_t mb = 0; mb < MBp; ++mb) {
            uint8_t byte = (mb < MB) ? s2d[mb * KB + k / BLOCK] : 0;
            int e = (int)byte - 127;
            for (int j = 0; j < BLOCK / 2; ++j) {
                int64_t m0 = mb * BLOCK + 2 * j, m1 = m0 + 1;
                double v0 = (m0 < M) ? oracle_bf16_to_f64(x[m0 * ldx + k]) : 0.0;
                double v1 = (m1 < M) ? oracle_bf16_to_f64(x[m1 * ldx + k]) : 0.0;
                uint8_t lo = oracle_e2m1_encode(ldexp(v0, -e));
                uint8_t hi = oracle_e2m1_encode(ldexp(v1, -e));
                q[k * (Mp / 2) + mb * (BLOCK / 2) + j] = (uint8_t)(lo | (hi << 4));
            }
            s[k * MBp + mb] = byte;
        }
    free(s2d);
    return 0;
}

/* ---------------------------------------------------------------------------------------
 * Hadamard transform of the column blobs: `_quantize_input_dual` and `_quantize_grad_dual`
 * in primus_turbo_mxfp4_local.py set `colwise_use_rht` for activations and gradients (the
 * weights use 2-D blocks instead).  Those column blobs are exactly the two operands of the
 * wgrad GEMM dW = dY^T . X, whose reduction runs over M.  The pages name the flag only;
 * reading taken:
 *   - T = (1/4) H16 diag(s) is applied to every group of 16 consecutive elements of a
 *     zero-padded column of X (rows 16g .. 16g + 15, g = 0 .. Mp/16 - 1), H16 the Sylvester
 *     Hadamard matrix (H[i][j] = (-1)^popcount(i & j)) and s a sign vector given by the
 *     caller as a 16-bit mask (bit j set: s_j = -1), the same for every group, both
 *     operands of a GEMM and every tensor of a step.  T^T T = I exactly (1/4 is a power of
 *     two), so (T dY)^T (T X) = dY^T X in exact arithmetic.
 *   - Order of the arithmetic, in fp32 with round-to-nearest-even at every step: each
 *     element is converted from bf16 (exact) and its sign flipped by s (exact); then the
 *     Walsh-Hadamard butterflies for h = 1, 2, 4, 8 in turn, each pair (j, j + h) with bit h
 *     of j clear becoming (v_j + v_{j+h}, v_j - v_{j+h}); then a multiplication by 0.25.
 *   - The 32-element MX blocks of the transformed column (two groups each) are quantized by
 *     the 1 x 32 rule above from these fp32 values.  Padding positions (rows M .. Mp - 1)
 *     are quantized from their transformed values too: a group that straddles M spreads its
 *     zeros, and keeping them makes the wgrad sum over all Mp positions equal the sum over
 *     the M real ones.
 *   - The transformed values must be finite (|x| < 2^124 is enough); otherwise the
 *     quantizer returns -1.
 * -------------------------------------------------------------------------------------- */

/* The 16-point transform of v, in place (order and precision as described above). */
void oracle_rht16(float v[16], uint32_t signs) {
    for (int j = 0; j < 16; ++j)
        if ((signs >> j) & 1u) v[j] = -v[j];
    for (int h = 1; h < 16; h <<= 1)
        for (int j = 0; j < 16; ++j)
            if (!(j & h)) {
                float a = v[j], b = v[j + h];
                v[j] = a + b;
                v[j + h] = a - b;
            }
    for (int j = 0; j < 16; ++j) v[j] = v[j] * 0.25f;
}

/* Col blob of X[M,K] with the transform applied along M; layout as oracle_quantize_col. */
int oracle_quantize_col_rht(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, uint32_t signs, uint8_t* q,
                            uint8_t* s) {
    int64_t Mp = cdiv64(M, PAD) * PAD, MBp = Mp / BLOCK;
    float* col = (float*)malloc((size_t)Mp * sizeof(float));
    if (!col) return -2;
    for (int64_t k = 0; k < K; ++k) {
        for (int64_t m = 0; m < Mp; ++m) col[m] = (m < M) ? (float)oracle_bf16_to_f64(x[m * ldx + k]) : 0.0f;
        for (int64_t g = 0; g < Mp / 16; ++g) oracle_rht16(col + 16 * g, signs);
        for (int64_t mb = 0; mb < MBp; ++mb) {
            double v[BLOCK];
            for (int i = 0; i < BLOCK; ++i) v[i] = (double)col[mb * BLOCK + i];
            if (quantize_block(v, q + k * (Mp / 2) + mb * (BLOCK / 2), &s[k * MBp + mb])) {
                free(col);
                return -1;
            }
        }
    }
    free(col);
    return 0;
}

/* The gradient recipe of `_quantize_grad_dual` with `use_sr` set: `colwise_use_rht` and
 * `colwise_use_sr` together.  Col blob of X[M,K] with the transform applied along M as in
 * oracle_quantize_col_rht, each 32-element block of the transformed column then quantized
 * with stochastic rounding as in oracle_quantize_col_sr: the scale byte from the block's
 * transformed values by the round-to-nearest rule, each scaled transformed element
 * rounded up or down by its 16 random bits, which are those of the blob position (row a =
 * column of X, column b = position along the padded M; packing 1).  col_ids (may be NULL):
 * the column index of each of the K columns in the full tensor. */
int oracle_quantize_col_rht_sr(const uint16_t* x, int64_t M, int64_t K, int64_t ldx, uint32_t signs, uint8_t* q,
                               uint8_t* s, uint64_t seed, const int64_t* col_ids) {
    int64_t Mp = cdiv64(M, PAD) * PAD, MBp = Mp / BLOCK;
    float* col = (float*)malloc((size_t)Mp * sizeof(float));
    if (!col) return -2;
    for (int64_t k = 0; k < K; ++k) {
        for (int64_t m = 0; m < Mp; ++m) col[m] = (m < M) ? (float)oracle_bf16_to_f64(x[m * ldx + k]) : 0.0f;
        for (int64_t g = 0; g < Mp / 16; ++g) oracle_rht16(col + 16 * g, signs);
        for (int64_t mb = 0; mb < MBp; ++mb) {
            double v[BLOCK];
            for (int i = 0; i < BLOCK; ++i) v[i] = (double)col[mb * BLOCK + i];
            if (quantize_block_sr(v, q + k * (Mp / 2) + mb * (BLOCK / 2), &s[k * MBp + mb], seed,
                                  col_ids ? col_ids[k] : k, mb * BLOCK, 1)) {
                free(col);
                return -1;
            }
        }
    }
    free(col);
    return 0;
}

/* ---------------------------------------------------------------------------------------
 * QK RMSNorm + interleaved RoPE backward, the producer computed in the quantizer's staging
 * read: the pages' MXFP6 QKV packer prologue (`MXFP6QKVNormRopeFunction`, whose packer
 * produces d(mixed_qkv) while staging its input; fused_norm_rope.py: the QK RMSNorm and an
 * interleaved RoPE rotation, per head q and k 3D columns apart in mixed_qkv, v passed
 * through unchanged).  Reading taken (the pages name the ops, not their formulas):
 *   - mixed_qkv[M, H*3*D]: for token m and head h, columns h*3D .. h*3D+D-1 are q, the next
 *     D are k, the next D are v;
 *   - forward for p in {q, k}: x = mixed[m, h, p, :]; r = 1/sqrt(mean(x^2) + eps) (saved by
 *     the forward); n = x r; y = n * w_p (w_q, w_k: the norm weights, [D]); interleaved RoPE
 *     on pairs (2i, 2i+1) with c = cos[m, i], s = sin[m, i]:
 *     o[2i] = y[2i] c - y[2i+1] s,  o[2i+1] = y[2i] s + y[2i+1] c;  v passes through;
 *   - backward, given g = dL/do in the same layout and the saved r:
 *     dy[2i] = g[2i] c + g[2i+1] s,  dy[2i+1] = -g[2i] s + g[2i+1] c;  dn = dy * w;
 *     dx = r dn - (r^3 / D) x sum_j(dn_j x_j);  d(mixed) for v is g itself.
 *     (dx is the derivative of o through n = x r(x); the norm weights' own gradient is a
 *     separate reduction, not part of d(mixed_qkv).)
 * The forward is here only to pin the backward (a numerical derivative of it); the product
 * computes the backward alone.
 * -------------------------------------------------------------------------------------- */

/* Forward of the norm + RoPE over mixed[M, H*3*D] (fp64 values): out in the same layout (v
 * copied), r_out[M, H, 2] the saved 1/sqrt(mean(x^2) + eps) of q and k. */
void oracle_qk_norm_rope_fwd(const double* mixed, const double* wq, const double* wk, const double* cosv,
                             const double* sinv, double eps, int64_t M, int64_t H, int64_t D, double* out,
                             double* r_out) {
    const int64_t ld = 3 * H * D;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t h = 0; h < H; ++h) {
            for (int p = 0; p < 2; ++p) {
                const double* x = mixed + m * ld + h * 3 * D + p * D;
                const double* w = p == 0 ? wq : wk;
                double* o = out + m * ld + h * 3 * D + p * D;
                double ss = 0.0;
                for (int64_t j = 0; j < D; ++j) ss += x[j] * x[j];
                const double r = 1.0 / sqrt(ss / (double)D + eps);
                r_out[(m * H + h) * 2 + p] = r;
                for (int64_t i = 0; i < D / 2; ++i) {
                    const double c = cosv[m * (D / 2) + i], sn = sinv[m * (D / 2) + i];
                    const double y0 = x[2 * i] * r * w[2 * i], y1 = x[2 * i + 1] * r * w[2 * i + 1];
                    o[2 * i] = y0 * c - y1 * sn;
                    o[2 * i + 1] = y0 * sn + y1 * c;
                }
            }
            for (int64_t j = 0; j < D; ++j) out[m * ld + h * 3 * D + 2 * D + j] = mixed[m * ld + h * 3 * D + 2 * D + j];
        }
}

/* Backward: g and x bf16 [M, H*3*D] (x = mixed_qkv, the forward's input), r[M, H, 2] (fp32,
 * as saved), w_q / w_k [D] and cos / sin [M, D/2] (fp32); out: d(mixed_qkv) [M, H*3*D] in
 * fp64. */
void oracle_qk_norm_rope_bwd(const uint16_t* g, const uint16_t* x, const float* r, const float* wq,
                             const float* wk, const float* cosv, const float* sinv, int64_t M, int64_t H,
                             int64_t D, double* out) {
    const int64_t ld = 3 * H * D;
    double* dn = (double*)malloc((size_t)D * sizeof(double));
    if (!dn) return;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t h = 0; h < H; ++h) {
            for (int p = 0; p < 2; ++p) {
                const int64_t base = m * ld + h * 3 * D + p * D;
                const float* w = p == 0 ? wq : wk;
                const double rr = (double)r[(m * H + h) * 2 + p];
                for (int64_t i = 0; i < D / 2; ++i) {
                    const double c = (double)cosv[m * (D / 2) + i], sn = (double)sinv[m * (D / 2) + i];
                    const double g0 = oracle_bf16_to_f64(g[base + 2 * i]), g1 = oracle_bf16_to_f64(g[base + 2 * i + 1]);
                    dn[2 * i] = (g0 * c + g1 * sn) * (double)w[2 * i];
                    dn[2 * i + 1] = (-g0 * sn + g1 * c) * (double)w[2 * i + 1];
                }
                double dot = 0.0;
                for (int64_t j = 0; j < D; ++j) dot += dn[j] * oracle_bf16_to_f64(x[base + j]);
                for (int64_t j = 0; j < D; ++j)
                    out[base + j] = rr * dn[j] - rr * rr * rr / (double)D * oracle_bf16_to_f64(x[base + j]) * dot;
            }
            for (int64_t j = 0; j < D; ++j) {
                const int64_t k = m * ld + h * 3 * D + 2 * D + j;
                out[k] = oracle_bf16_to_f64(g[k]);
            }
        }
    free(dn);
}

