/*
 * mxfp4.h -- C ABI of the GB300 (sm_103a) MXFP4 linear hot path.
 *
 * Three operations, all enqueued asynchronously on a caller stream:
 *   mxfp4_quantize       row-only quantizer (forward-only regions)
 *   mxfp4_quantize_dual  rowwise + columnwise quantizer from one read of the input
 *   mxfp4_gemm           block-scaled MXF4 GEMM  C[M,N] = A[M,K] . B[N,K]^T
 *
 * Formats (primus_turbo_mxfp4_local.py, `_quantize_mxfp4_dual_fake`, non-shuffled
 * branch, and module constants MXFP4_BLOCK_SIZE = 32, MXFP4_PADDING_ALIGN_SIZE = 128):
 *   - Input: bf16 X[M,K], row-major with a row pitch of ldx elements.
 *   - Kp = ceil(K/128)*128 and Mp = ceil(M/128)*128: only the packed dimension is padded.
 *   - Row blob of X: elements q[M, Kp/2] (FP4 E2M1, two per byte, element 2j in the low
 *     nibble of byte j) and one E8M0 scale byte per 32-element block along K.
 *   - Col blob of X: the row blob of X^T, q[K, Mp/2] plus its scales.  It is what the
 *     dgrad (dX = dY . W: B = col blob of W) and wgrad (dW = dY^T . X: A = col blob of
 *     dY, B = col blob of X) GEMMs of `MXFP4LinearFunction.backward` consume.
 *   - Padding elements are +0 and all-padding blocks have the scale byte 0x00.
 *   - Quantization rule (OCP MX v1.0 for MXFP4; the pages print no formula): scale
 *     exponent e = floor(log2(amax)) - 2 clamped to [-127, 127] (byte e + 127; an
 *     all-zero block gets 0x00), element = round-to-nearest-even of v / 2^e onto
 *     {0, 0.5, 1, 1.5, 2, 3, 4, 6}, saturating at 6, sign kept (also for zero).
 *     Inputs must be finite; non-finite inputs give unspecified bytes.
 *
 * Scale layouts (mxfp4_scale_layout):
 *   MXFP4_SCALE_PLAIN  s[R, KB] row-major, R = rows of the blob, KB = (packed dim)/32.
 *                      Same shape as the pages' non-shuffled scale tensors.
 *   MXFP4_SCALE_TC     the layout the tcgen05 block-scaled MMA reads: rows padded to a
 *                      multiple of 128 (padding bytes 0x00), cut into 128-row x 4-block
 *                      atoms of 512 bytes, atoms ordered block-group fastest
 *                      (atom = (r/128) * (KB/4) + kb/4); in an atom byte (r, kb) is at
 *                      (r%32)*16 + ((r%128)/32)*4 + kb%4.  Size ceil(R/128)*128*KB bytes.
 *                      mxfp4_gemm requires this layout.  It replaces the pages'
 *                      MI355X preshuffle, which needed extra shuffle launches per GEMM;
 *                      here the quantizer writes it directly.
 *
 * Ownership: the caller allocates every buffer (use mxfp4_quantize_sizes); the library
 * never allocates, frees or synchronizes on these calls.  Buffers must be device memory
 * on the current device.
 *
 * Errors: argument, alignment and device checks run on the host before anything is
 * enqueued and return a status without touching the buffers.  Every kernel wait is
 * bounded; a wait that runs out records a device-side error word that
 * mxfp4_last_device_error reports.  There is no fallback path: on an unsupported device
 * the calls fail with MXFP4_ERR_UNSUPPORTED_DEVICE.
 */
#ifndef MXFP4_GB300_H
#define MXFP4_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t; NULL selects the legacy default stream. */
typedef struct CUstream_st* mxfp4_stream_t;

typedef enum {
    MXFP4_OK = 0,
    MXFP4_ERR_INVALID_ARG = 1,        /* a size, pitch, pointer or enum is out of range   */
    MXFP4_ERR_MISALIGNED = 2,         /* a pointer or pitch breaks the 16-byte rule       */
    MXFP4_ERR_UNSUPPORTED_DEVICE = 3, /* current device is not compute capability 10.3    */
    MXFP4_ERR_CUDA = 4,               /* a CUDA runtime/driver call or a launch failed    */
    MXFP4_ERR_TIMEOUT = 5,            /* a kernel's bounded wait ran out (device word)    */
    MXFP4_ERR_NONFINITE = 6           /* a tensorwise FP8 amax was NaN or inf (device word) */
} mxfp4_status;

typedef enum { MXFP4_SCALE_PLAIN = 0, MXFP4_SCALE_TC = 1 } mxfp4_scale_layout;

typedef enum { MXFP4_OUT_BF16 = 0, MXFP4_OUT_F32 = 1 } mxfp4_out_dtype;

/* Bytes of the element buffer and of the scale buffer of one blob with `rows` rows and a
 * packed dimension of logical length `k` (padded to Kp = ceil(k/128)*128):
 * q_bytes = rows * Kp/2; s_bytes = rows * Kp/32 (PLAIN) or ceil(rows/128)*128 * Kp/32
 * (TC).  For the row blob of X[M,K] pass (M, K); for the col blob pass (K, M).
 * Either output pointer may be NULL.  rows, k >= 1, else MXFP4_ERR_INVALID_ARG. */
mxfp4_status mxfp4_quantize_sizes(int64_t rows, int64_t k, mxfp4_scale_layout layout,
                                  size_t* q_bytes, size_t* s_bytes);

/* Row-only quantizer: the row blob of X (primus_turbo_mxfp4_local.py calls
 * `quantize_mxfp4`; the row-only rationale is the "row-only packing" paragraph of Primus
 * PR #1107: column blobs only feed backward, so forward-only regions skip them).
 *   x      bf16 X[M,K], row pitch ldx elements (ldx >= K, ldx % 8 == 0), 16-byte aligned
 *   q_row  out, M * Kp/2 bytes;  s_row  out, scale bytes in `layout`
 * All of q_row and s_row (padding included) is written.  M, K >= 1. */
mxfp4_status mxfp4_quantize(const void* x, int64_t M, int64_t K, int64_t ldx, void* q_row,
                            void* s_row, mxfp4_scale_layout layout, mxfp4_stream_t stream);

/* Dual quantizer: row blob and col blob of X from one read of X (primus_turbo_mxfp4_local.py,
 * `_quantize_mxfp4_dual_op` with every recipe and shuffle flag off; outputs in the order
 * row_q, row_s, col_q, col_s).
 *   q_col  out, K * Mp/2 bytes;  s_col  out, col-blob scale bytes in `layout`
 * Other arguments as mxfp4_quantize. */
mxfp4_status mxfp4_quantize_dual(const void* x, int64_t M, int64_t K, int64_t ldx,
                                 void* q_row, void* s_row, void* q_col, void* s_col,
                                 mxfp4_scale_layout layout, mxfp4_stream_t stream);

/* Dual quantizer with stochastically rounded elements: the gradient quantization of
 * `_quantize_grad_dual` in primus_turbo_mxfp4_local.py with `use_sr` set (the
 * `rowwise_use_sr` / `colwise_use_sr` flags; the layer's
 * `mxfp4_gradient_stochastic_rounding` option), every other recipe flag off.  The pages
 * name the flag only; what it computes here:
 *   - scale bytes exactly as mxfp4_quantize_dual;
 *   - each scaled element y: |y| >= 6 gives 6; otherwise, with lo <= |y| < hi its
 *     neighbours on {0, .5, 1, 1.5, 2, 3, 4, 6}, hi if r < floor((|y| - lo)/(hi - lo) * 2^16)
 *     and lo otherwise, with the sign kept; r = 16 random bits of the element;
 *   - r: Philox4x32-10 keyed by `seed` (low word first), counter (b/8, a, packing, 0) for
 *     row a, column b of the blob (packing 0: row blob of X, a = row of X; 1: col blob,
 *     a = column of X), bits in word (b/2) % 4, low half for even b.
 * The same seed gives the same bytes; the caller picks a new seed per step.  Arguments
 * otherwise as mxfp4_quantize_dual. */
mxfp4_status mxfp4_quantize_dual_sr(const void* x, int64_t M, int64_t K, int64_t ldx,
                                    void* q_row, void* s_row, void* q_col, void* s_col,
                                    mxfp4_scale_layout layout, uint64_t seed,
                                    mxfp4_stream_t stream);

/* Dual quantizer with 2-D block scales: the weight quantization of `_quantize_weight_dual`
 * in primus_turbo_mxfp4_local.py (`rowwise_use_2d_block` and `colwise_use_2d_block` set,
 * every other recipe flag off).  The pages name the flags only; what it computes here: X
 * is cut into 32 x 32 blocks (padding +0), each block gets one E8M0 scale byte from the
 * amax of its 1024 elements by the rule above, and every element of the block is encoded
 * with that scale in both packings -- so the row blob's scale of (row r, block kb) and the
 * col blob's scale of (column k, block mb) are the scale of the 2-D block that holds them,
 * and the two blobs dequantize to exact transposes of each other.  Scale bytes of padding
 * rows of the tensor-core layout are 0x00, as for the 1-D blobs.  Arguments, layouts and
 * errors as mxfp4_quantize_dual. */
mxfp4_status mxfp4_quantize_dual_2d(const void* x, int64_t M, int64_t K, int64_t ldx,
                                    void* q_row, void* s_row, void* q_col, void* s_col,
                                    mxfp4_scale_layout layout, mxfp4_stream_t stream);

/* Dual quantizer with the Hadamard transform of the column blob: the activation and
 * gradient quantization of `_quantize_input_dual` / `_quantize_grad_dual` in
 * primus_turbo_mxfp4_local.py with `colwise_use_rht` set (every other recipe flag off).
 * The pages name the flag only; what it computes here: the row blob exactly as
 * mxfp4_quantize_dual; for the col blob, every group of 16 consecutive elements along M of
 * a zero-padded column of X (rows 16g .. 16g + 15 up to Mp) becomes T x with
 * T = (1/4) H16 diag(s) -- H16 the Sylvester Hadamard matrix, H[i][j] = (-1)^popcount(i & j),
 * s_j = -1 where bit j of `signs` is set -- computed in fp32 with round-to-nearest-even:
 * signs applied, butterflies (v_j, v_j+h) -> (v_j + v_j+h, v_j - v_j+h) for h = 1, 2, 4, 8
 * in turn, then x 0.25; each 32-element block of the transformed column is quantized by
 * the rule above from those fp32 values, padding positions included (a group straddling M
 * spreads its zeros; keeping them makes a GEMM over all Mp positions exact).  T^T T = I,
 * so dW = dY^T . X is unchanged in exact arithmetic when both col blobs use the same
 * signs.  Transformed values must be finite (|x| < 2^124 suffices).  Arguments, layouts
 * and errors as mxfp4_quantize_dual; signs: bits 0..15. */
mxfp4_status mxfp4_quantize_dual_rht(const void* x, int64_t M, int64_t K, int64_t ldx,
                                     void* q_row, void* s_row, void* q_col, void* s_col,
                                     mxfp4_scale_layout layout, uint32_t signs,
                                     mxfp4_stream_t stream);

/* The full gradient quantization of `_quantize_grad_dual` in primus_turbo_mxfp4_local.py
 * with `use_sr` set: `rowwise_use_sr`, `colwise_use_sr` and `colwise_use_rht` together.
 * The row blob exactly as mxfp4_quantize_dual_sr; the col blob transformed exactly as in
 * mxfp4_quantize_dual_rht, each 32-element block of the transformed column then getting
 * the round-to-nearest scale byte of its transformed values and stochastically rounded
 * elements by the rule of mxfp4_quantize_dual_sr, with the random bits of the element's
 * col-blob position (row a = column of X, column b = position along the padded M,
 * packing 1).  Arguments, layouts and errors as mxfp4_quantize_dual; signs: bits 0..15;
 * seed as mxfp4_quantize_dual_sr. */
mxfp4_status mxfp4_quantize_dual_rht_sr(const void* x, int64_t M, int64_t K, int64_t ldx,
                                        void* q_row, void* s_row, void* q_col, void* s_col,
                                        mxfp4_scale_layout layout, uint32_t signs, uint64_t seed,
                                        mxfp4_stream_t stream);

/* The gradient quantization of the QKV projection with the QK RMSNorm + interleaved RoPE
 * backward computed in the quantizer's staging read: the prologue of the pages' QKV packer
 * (`MXFP6QKVNormRopeFunction`, whose packer produces d(mixed_qkv) while staging its input, so
 * the norm + RoPE backward never writes it to HBM for the quantizer to read again;
 * fused_norm_rope.py: per head, q and k are 3D columns apart in mixed_qkv, the rotation acts
 * on interleaved pairs, v passes through unchanged).  Head dimension 128.  With K = 3*H*128:
 *   g       bf16 [M, K]: the gradient of the norm + RoPE output, per token and head the
 *           columns h*384 .. h*384+127 for q, the next 128 for k, the next 128 for v (v's
 *           gradient itself); row pitch K
 *   x       bf16 [M, K]: mixed_qkv, the projection's output the forward normalized (same
 *           layout; only its q and k columns are read)
 *   rstd    fp32 [M, H, 2]: the forward's 1/sqrt(mean(x^2) + eps) of q (0) and k (1)
 *   wq, wk  fp32 [128]: the norm weights; cos_table, sin_table fp32 [M, 64]: the RoPE angles
 *           of each token, pair i rotating elements (2i, 2i+1)
 * What is quantized: d(mixed_qkv)[M, K] with, for q and k, dy = the inverse rotation of g,
 * dn = dy * w, dx = r dn - (r^3/128) x sum(dn x), computed in fp32 and rounded once to bf16
 * (to nearest even), and for v the gradient g; the outputs are exactly those of
 * mxfp4_quantize_dual over that bf16 d(mixed_qkv), which is also written to `dmixed`
 * (bf16 [M, K], pitch K) when it is not NULL.  Alignment: g, x, cos_table, sin_table and
 * dmixed 16 bytes, rstd, wq, wk 4 bytes; blobs and layouts as mxfp4_quantize_dual.  H >= 1;
 * errors as mxfp4_quantize_dual. */
mxfp4_status mxfp4_quantize_dual_qk_norm_rope_bwd(const void* g, const void* x, int64_t M, int64_t H,
                                                  const float* rstd, const float* wq, const float* wk,
                                                  const float* cos_table, const float* sin_table,
                                                  void* q_row, void* s_row, void* q_col, void* s_col,
                                                  mxfp4_scale_layout layout, void* dmixed,
                                                  mxfp4_stream_t stream);

/* Bits of mxfp4_quantize_task::flags. */
#define MXFP4_QUANT_2D_BLOCKS 1   /* 32 x 32 blocks, as mxfp4_quantize_dual_2d (row-only too) */
#define MXFP4_QUANT_RHT_COL 2     /* col blob transformed, as mxfp4_quantize_dual_rht (dual only) */

/* One tensor of a batched quantization: bf16 x[rows, k] with row pitch ldx elements and
 * its output buffers, as for mxfp4_quantize / mxfp4_quantize_dual (q_col and s_col are
 * read only for the dual quantizer); flags: 0, MXFP4_QUANT_2D_BLOCKS or
 * MXFP4_QUANT_RHT_COL (not both); rht_signs: the sign mask of MXFP4_QUANT_RHT_COL;
 * amax (row-only batches, dual == 0; MXFP4_ERR_INVALID_ARG otherwise): NULL, or one fp32
 * in device memory (4-byte aligned) that the call sets to max |x| over the tensor, the amax
 * of the tensorwise FP8 quantizer (mxfp4_fp8_quantize_tw), from the block maxima the
 * rowwise pass takes anyway: the hybrid backward's FP8 quantization of X and W, whose
 * forward is row-only, then skips its own amax pass (mxfp4_fp8_quantize_task::amax_given).
 * A NaN or infinity in x makes it non-finite, as there. */
typedef struct {
    const void* x;
    int64_t rows;
    int64_t k;
    int64_t ldx;
    void* q_row;
    void* s_row;
    void* q_col;
    void* s_col;
    int32_t flags;
    uint32_t rht_signs;
    float* amax;
} mxfp4_quantize_task;

#define MXFP4_MAX_BATCH 4

/* Quantizes 1..MXFP4_MAX_BATCH independent tensors in one launch, each with exactly the
 * output of mxfp4_quantize (dual == 0) or mxfp4_quantize_dual (dual != 0), or with a task
 * flag that of mxfp4_quantize_dual_2d / mxfp4_quantize_dual_rht.  Same
 * operation as those two (the per-tensor `quantize_mxfp4` / `_quantize_mxfp4_dual_op`
 * calls of primus_turbo_mxfp4_local.py); one launch lets a small tensor share the GPU with
 * a large one instead of paying its own ramp-up and tail (the forward step quantizes X and
 * W together).  Tasks must not overlap in memory.  Every task is checked before anything
 * runs: the first failing task's status is returned and nothing is launched. */
mxfp4_status mxfp4_quantize_batch(int32_t count, const mxfp4_quantize_task* tasks, int32_t dual,
                                  mxfp4_scale_layout layout, mxfp4_stream_t stream);

/* Block-scaled GEMM C[M,N] = A . B^T over two K-packed blobs (the "TN" form that the
 * forward, dgrad and wgrad `gemm_fp4_impl` calls of `MXFP4LinearFunction` reduce to):
 *   a_q  A elements [M, Kp/2];  a_s  A scales, MXFP4_SCALE_TC layout for (M, K)
 *   b_q  B elements [N, Kp/2];  b_s  B scales, MXFP4_SCALE_TC layout for (N, K)
 *   K    logical reduction length (Kp = ceil(K/128)*128 is what the blobs hold; padding
 *        is zero, so the sum over Kp equals the sum over K)
 *   c    out, C[M,N] row-major with pitch ldc elements (ldc >= N), bf16 or fp32
 * Products of the dequantized elements accumulate in fp32 on the tensor cores; bf16
 * output is rounded once, to nearest even.  All pointers 16-byte aligned.  M, N, K >= 1.
 */
mxfp4_status mxfp4_gemm(const void* a_q, const void* a_s, const void* b_q, const void* b_s,
                        int64_t M, int64_t N, int64_t K, void* c, int64_t ldc,
                        mxfp4_out_dtype out_dtype, mxfp4_stream_t stream);

/* mxfp4_gemm followed by the layer's bias add, in the same launch: the `output + bias`
 * of `_forward_impl` in MXFP4ColumnParallelLinear / MXFP4RowParallelLinear
 * (primus_turbo_mxfp4_local.py), which adds the bf16 bias vector to every row of the GEMM
 * output.  C[m,n] = out(out(A.B^T [m,n]) + bias[n]) with the same two roundings as the
 * unfused pair of operations: out() rounds to the output dtype to nearest even, and the
 * add itself is done in fp32 (bf16 output: the GEMM result is rounded to bf16 first;
 * fp32 output: the fp32 sum).
 *   bias  bf16[N], 16-byte aligned, not NULL (MXFP4_ERR_INVALID_ARG); read only.
 * Everything else as mxfp4_gemm. */
mxfp4_status mxfp4_gemm_bias(const void* a_q, const void* a_s, const void* b_q, const void* b_s,
                             int64_t M, int64_t N, int64_t K, const void* bias, void* c,
                             int64_t ldc, mxfp4_out_dtype out_dtype, mxfp4_stream_t stream);

/* A forward GEMM whose epilogue also quantizes its output for the next linear layer: the
 * fusion that emits the next layer's MXFP4 blobs from the GEMM epilogue, in the layer chain
 * (`MXFP4LinearFunction.forward` of primus_turbo_mxfp4_local.py feeds each layer's output
 * to the next layer, whose forward starts with `_quantize_mxfp4_dual_op` of that output).
 * Writes bf16 C = A . B^T (+ bias), exactly as mxfp4_gemm / mxfp4_gemm_bias with
 * MXFP4_OUT_BF16, and the MXFP4 blobs of C's bf16 values exactly as
 * mxfp4_quantize_dual(C) (q_col and s_col set) or mxfp4_quantize(C) (both NULL) with
 * MXFP4_SCALE_TC would write them, padding included:
 *   q_row [M, Np/2], s_row  the row blob of C (blocks of 32 along N), Np = ceil(N/128)*128
 *   q_col [N, Mp/2], s_col  the col blob of C (blocks of 32 along M), Mp = ceil(M/128)*128
 * C is not read back: the blobs come from the accumulator tile after its bf16 rounding,
 * in the epilogue of the CTA-pair kernel (one extra launch, the quantizer over C, when M is
 * at most 128).  bias: bf16[N] or NULL.  ldc: a multiple of 8 (MXFP4_ERR_MISALIGNED
 * otherwise, as for an unaligned pointer); q_row, s_row not NULL, q_col and s_col both
 * NULL or both set (MXFP4_ERR_INVALID_ARG).  Everything else as mxfp4_gemm. */
mxfp4_status mxfp4_gemm_quantize(const void* a_q, const void* a_s, const void* b_q, const void* b_s,
                                 int64_t M, int64_t N, int64_t K, const void* bias, void* c, int64_t ldc,
                                 void* q_row, void* s_row, void* q_col, void* s_col,
                                 mxfp4_stream_t stream);

/* One GEMM of a batch: the arguments of mxfp4_gemm, and an optional bias (NULL: none;
 * otherwise as for mxfp4_gemm_bias). */
typedef struct {
    const void* a_q;
    const void* a_s;
    const void* b_q;
    const void* b_s;
    int64_t M;
    int64_t N;
    int64_t K;
    void* c;
    int64_t ldc;
    mxfp4_out_dtype out_dtype;
    const void* bias;
} mxfp4_gemm_task;

/* 1..MXFP4_MAX_BATCH independent GEMMs, each with exactly the result its own mxfp4_gemm
 * call gives (the dgrad and wgrad `gemm_fp4_impl` calls of
 * `MXFP4LinearFunction.backward` read the same quantized dY and run back to back).  The
 * problems with more than one 128-row tile share one launch, whose CTA pairs walk the
 * tiles of all of them, so neither pays its own ramp-up and tail.  Outputs must not
 * overlap each other or any input.  Every task is checked before anything runs: the first
 * failing task's status is returned and nothing is launched. */
mxfp4_status mxfp4_gemm_batch(int32_t count, const mxfp4_gemm_task* tasks, mxfp4_stream_t stream);

/* Output tile width of the CTA-pair GEMM launches (problems of more than one 128-row tile)
 * made by the calls that follow, process-wide:
 *   MXFP4_TILES_AUTO    (the default) each launch takes the width whose modelled time is
 *                       lower: the tiles dealt round-robin to the co-resident CTA pairs,
 *                       each costing its K steps and an accumulator hand-over;
 *   MXFP4_TILES_NARROW  256 x 256 tiles;
 *   MXFP4_TILES_WIDE    256 x 384 tiles (a sixth fewer operand bytes per flop and a third
 *                       fewer hand-overs, at a coarser tile grid) wherever the launch
 *                       allows them: every pair problem of the launch with bf16 output and
 *                       a pitch that is a multiple of 8 elements; other launches narrow.
 * The width changes no result: the same bits come out either way (the tests check this).
 * mxfp4_gemm_quantize always runs narrow tiles.  An unknown policy returns
 * MXFP4_ERR_INVALID_ARG and changes nothing. */
#define MXFP4_TILES_AUTO 0
#define MXFP4_TILES_NARROW 1
#define MXFP4_TILES_WIDE 2
mxfp4_status mxfp4_gemm_set_tile_policy(int32_t policy);

/* ---- hybrid FP8 backward --------------------------------------------------------------
 * `MXFP4LinearFunction.backward` in primus_turbo_mxfp4_local.py, when the layer's
 * `mxfp4_backward_precision` is "fp8" (`backward_is_fp8`): dY, X and W are quantized
 * tensorwise to FP8 E5M2 (`_quantize_fp8_tw(…, float8_e5m2)`) and dgrad / wgrad run as
 * FP8 GEMMs with TENSORWISE scales (`gemm_fp8_impl`).  The forward stays MXFP4. */

/* Tensorwise E5M2 quantization of bf16 X[M,K].  The pages call `_quantize_fp8_tw` without
 * defining it; what it computes here:
 *   amax = max |x| over the tensor;  scale = 57344 / amax in fp32 (57344 = the largest
 *   finite E5M2 value; the largest finite fp32 if the quotient overflows; 1 if amax = 0);
 *   element = E5M2 round-to-nearest-even of the fp32 product x * scale, saturating at
 *   +-57344, sign of zero kept;  scale_inv = 1 / scale in fp32.
 *   x          bf16 X[M,K], row pitch ldx elements (ldx >= K, ldx % 8 == 0), 16-byte aligned
 *   q_row      out or NULL: X's codes, M rows of round16(K) bytes (padding bytes 0x00)
 *   q_col      out or NULL: X^T's codes, K rows of round16(M) bytes (padding 0x00); at
 *              least one of q_row / q_col; both 16-byte aligned
 *   amax, scale_inv   out, one fp32 each in device memory (4-byte aligned); the GEMMs
 *              read scale_inv from there, so no host synchronization is needed.
 * Launches on `stream`: *amax zeroed, an amax pass, the conversion.  M, K >= 1.
 * Inputs must be finite: a NaN or infinity makes amax non-finite, the codes and scale_inv
 * of that tensor are then meaningless, and the conversion records it in the device error
 * word (mxfp4_last_device_error returns MXFP4_ERR_NONFINITE). */
mxfp4_status mxfp4_fp8_quantize_tw(const void* x, int64_t M, int64_t K, int64_t ldx,
                                   void* q_row, void* q_col, float* amax, float* scale_inv,
                                   mxfp4_stream_t stream);

/* One tensor of a batch: the arguments of mxfp4_fp8_quantize_tw; amax_given nonzero: *amax
 * already holds max |x| of this tensor (written by an earlier mxfp4_quantize_batch amax
 * output, in stream order before this call) and the call neither zeroes it nor runs the
 * amax pass over the tensor. */
typedef struct {
    const void* x;
    int64_t M;
    int64_t K;
    int64_t ldx;
    void* q_row;
    void* q_col;
    float* amax;
    float* scale_inv;
    int32_t amax_given;
} mxfp4_fp8_quantize_task;

/* 1..MXFP4_MAX_BATCH tensors quantized tensorwise with the same three launches (the hybrid
 * backward quantizes dY, X and W together), each with exactly its own call's result.
 * Tasks must not overlap in memory.  Every task is checked before anything runs. */
mxfp4_status mxfp4_fp8_quantize_tw_batch(int32_t count, const mxfp4_fp8_quantize_task* tasks,
                                         mxfp4_stream_t stream);

/* FP8 GEMM C[M,N] = (A . B^T) * (*a_scale_inv) * (*b_scale_inv) over E5M2 codes, the form
 * both backward `gemm_fp8_impl` calls take with the quantizer's column copies (dgrad:
 * A = dY row copy, B = W column copy; wgrad: A = dY column copy, B = X column copy):
 *   a   [M, round16(K)] codes;  b   [N, round16(K)] codes (16-byte aligned; bytes past K
 *       are not read)
 *   a_scale_inv, b_scale_inv   device fp32 (as mxfp4_fp8_quantize_tw leaves them)
 *   c   out, C[M,N] row-major with pitch ldc elements (ldc >= N), bf16 or fp32
 * Products accumulate in fp32 on the tensor cores; the accumulator is multiplied by the
 * fp32 product of the two inverse scales and rounded once to the output dtype.
 * M, N, K >= 1. */
mxfp4_status mxfp4_fp8_gemm(const void* a, const float* a_scale_inv, const void* b,
                            const float* b_scale_inv, int64_t M, int64_t N, int64_t K, void* c,
                            int64_t ldc, mxfp4_out_dtype out_dtype, mxfp4_stream_t stream);

/* One FP8 GEMM of a batch: the arguments of mxfp4_fp8_gemm. */
typedef struct {
    const void* a;
    const float* a_scale_inv;
    const void* b;
    const float* b_scale_inv;
    int64_t M;
    int64_t N;
    int64_t K;
    void* c;
    int64_t ldc;
    mxfp4_out_dtype out_dtype;
} mxfp4_fp8_gemm_task;

/* 1..MXFP4_MAX_BATCH FP8 GEMMs in one launch of CTA pairs (dgrad and wgrad of the hybrid
 * backward together), each with exactly its own call's result.  Outputs must not overlap
 * each other or any input.  Every task is checked before anything runs. */
mxfp4_status mxfp4_fp8_gemm_batch(int32_t count, const mxfp4_fp8_gemm_task* tasks,
                                  mxfp4_stream_t stream);

/* ---- a step from host memory to host memory -------------------------------------------
 * The data path of `MXFP4LinearFunction` (primus_turbo_mxfp4_local.py) for linears whose
 * bf16 inputs and results live in host memory: per linear, forward = dual (train) or
 * row-only quantization of X and W and Y = X . W^T; backward = dual quantization of dY,
 * dX = dY . W and dW = dY^T . X.  The forwards run in task order and the backwards in
 * reverse task order, the order of a block's backward pass (Flux-12B's single-stream block:
 * linear1 then linear2 forward, linear2 then linear1 backward). */
typedef struct {
    const void* x;     /* host bf16 X[M,K], dense rows of K elements                     */
    const void* w;     /* host bf16 W[N,K], dense                                        */
    const void* dy;    /* host bf16 dY[M,N], dense (train); ignored otherwise            */
    void* y;           /* host out: Y[M,N] in out_dtype, dense                           */
    void* dx;          /* host out: dX[M,K] in out_dtype (train)                         */
    void* dw;          /* host out: dW[N,K] in out_dtype (train)                         */
    int64_t M;
    int64_t N;
    int64_t K;
    int32_t train;     /* 1: forward and backward; 0: forward only (row-only quantizer)   */
    mxfp4_out_dtype out_dtype;
} mxfp4_linear_host_task;

/* Bytes of device workspace mxfp4_linear_step_host needs for these tasks (the device
 * copies of the inputs, every blob, and the device results).  count in 1..MXFP4_MAX_BATCH;
 * only the shapes, out_dtype and train of each task are read (the pointers may be NULL). */
mxfp4_status mxfp4_linear_workspace_bytes(int32_t count, const mxfp4_linear_host_task* tasks,
                                          size_t* bytes);

/* Enqueues one step of `count` linears: host-to-device copies of every input, the
 * library's quantizer and GEMM kernels, and device-to-host copies of every result.
 *   workspace        caller-owned device memory of at least mxfp4_linear_workspace_bytes
 *                    (256-byte aligned); its contents are scratch between calls
 *   stream           the kernels run on it; the copies run on two streams the library
 *                    creates once per device (never freed), ordered against `stream` with
 *                    events, so copies overlap the kernels of other linears and the
 *                    quantizer of each linear waits only for its own inputs.  When the call
 *                    returns, `stream` is ordered after every copy: synchronizing it makes
 *                    the results visible in host memory.
 * Host buffers should be pinned (page-locked) for the copies to be asynchronous.  All
 * arguments are checked before anything is enqueued; a CUDA failure after that returns
 * MXFP4_ERR_CUDA and may leave part of the step enqueued.  Calls from several host threads
 * are serialized by the library (they share the copy streams). */
mxfp4_status mxfp4_linear_step_host(int32_t count, const mxfp4_linear_host_task* tasks,
                                    void* workspace, size_t workspace_bytes, mxfp4_stream_t stream);

/* Pipelined form of mxfp4_linear_step_host for a loop of steps: the same copies, kernels
 * and results, but consecutive calls overlap.  Each refill of a device input waits only for
 * the previous step's quantizer of that input, the results of consecutive steps leave from
 * two output sets used alternately, and when the call returns `stream` is ordered after the
 * step's kernels and copies in but NOT after its copies out, so the next step's copies in
 * and kernels run while this step's results are still being copied out.
 *   workspace  at least mxfp4_linear_pipelined_workspace_bytes (the plain step's workspace
 *              and a second output set), 256-byte aligned; keep the same workspace and
 *              tasks' shapes from one call to the next
 * The host results of a step are in host memory once mxfp4_linear_host_wait(stream) has
 * been called after it and `stream` has been synchronized.  A host input buffer may be
 * rewritten once `stream` has passed the call (its copies in are done); a host output
 * buffer is written by every call that names it, in call order.  Errors as for
 * mxfp4_linear_step_host.  A plain mxfp4_linear_step_host call between pipelined ones is
 * allowed (it waits for everything before it, as always). */
mxfp4_status mxfp4_linear_pipelined_workspace_bytes(int32_t count, const mxfp4_linear_host_task* tasks,
                                                    size_t* bytes);
mxfp4_status mxfp4_linear_step_host_pipelined(int32_t count, const mxfp4_linear_host_task* tasks,
                                              void* workspace, size_t workspace_bytes,
                                              mxfp4_stream_t stream);

/* Orders `stream` after every copy (in and out) of every host step enqueued on the current
 * device so far: synchronizing `stream` afterwards makes all their results visible in host
 * memory. */
mxfp4_status mxfp4_linear_host_wait(mxfp4_stream_t stream);

/* Synchronizes `stream`, then reads and clears the device error word of the current
 * device: MXFP4_ERR_TIMEOUT if a bounded wait in any kernel of this library ran out
 * since the last call, else MXFP4_ERR_NONFINITE if a tensorwise FP8 quantization met a
 * non-finite amax; MXFP4_ERR_CUDA if the synchronization itself failed; else OK. */
mxfp4_status mxfp4_last_device_error(mxfp4_stream_t stream);

/* Diagnostic for the bounded-wait machinery: launches one warp that waits on a barrier
 * nothing ever arrives at, with a limit of timeout_ns (1 .. 10^10 ns).  The wait runs out,
 * the kernel records the error word and returns, so a following mxfp4_last_device_error
 * must report MXFP4_ERR_TIMEOUT while the context stays usable. */
mxfp4_status mxfp4_selftest_bounded_wait(int64_t timeout_ns, mxfp4_stream_t stream);

/* Static, never NULL. */
const char* mxfp4_status_string(mxfp4_status status);

#ifdef __cplusplus
}
#endif

#endif /* MXFP4_GB300_H */
