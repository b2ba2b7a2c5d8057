// launch.h -- internal interface between the C ABI (api.cu) and the kernel translation
// units (quantize.cu, gemm.cu).  Not installed; the public interface is include/mxfp4.h.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace mxfp4 {

// ---- quantizer -------------------------------------------------------------------------
struct QuantArgs {
    int64_t M, K;        // logical shape of X
    int32_t tiles_m;     // ceil(M / 128)
    int32_t tiles_k;     // ceil(K / 128)
    uint8_t* q_row;      // [M, Kp/2]
    uint8_t* s_row;      // row-blob scales
    uint8_t* q_col;      // [K, Mp/2]   (dual only)
    uint8_t* s_col;      // col-blob scales (dual only)
    int64_t ldq_row;     // Kp / 2
    int64_t ldq_col;     // Mp / 2
    int64_t kb_row;      // Kp / 32
    int64_t kb_col;      // Mp / 32
    int32_t tc_layout;   // 1: tensor-core scale layout, 0: plain
    uint64_t seed;       // Philox key of the stochastic-rounding instance (unused otherwise)
    int32_t block_2d;    // 1: 32 x 32 blocks (one scale per block in both packings)
    int32_t rht;         // 1: Hadamard transform of 16-row groups before the column pass
    uint32_t rht_signs;  // its sign mask (bit j: row j of a group is negated)
    uint32_t* amax_bits; // or null: raised (atomic max) to max |x| as fp32 bits, zeroed before the launch
    uint32_t* err;       // device error word
};

// Up to kMaxQuantTasks independent tensors quantized by one launch; tile t of the launch
// belongs to the first task j with t < tile_end[j].  maps[j]: bf16 X of task j as a 2-D
// tensor {K, M} (innermost first), box {64, 128} with the 128-byte swizzle (a 128 x 128
// tile is two boxes), out-of-bounds elements read as zero.
constexpr int kMaxQuantTasks = 4;
struct QuantBatch {
    CUtensorMap maps[kMaxQuantTasks];
    QuantArgs args[kMaxQuantTasks];
    int32_t tile_end[kMaxQuantTasks];
    int32_t count;
};

// Dual quantization of d(mixed_qkv) computed in the staging read from the gradient of the
// QK RMSNorm + interleaved RoPE output (the quantizer prologue).  gmap / xmap: the gradient
// g and mixed_qkv x as bf16 2-D tensors {3*H*128, M} (box {64, 128}, 128-byte swizzle, zero
// fill); q: the quantization task for d(mixed_qkv) [M, 3*H*128] (dual).
constexpr int kNormRopeD = 128;   // head dimension
constexpr int kNormRopeMaxUnitHeads = 16;   // a unit of work touches at most this many heads
struct NormRopeArgs {
    CUtensorMap gmap;
    CUtensorMap xmap;
    QuantArgs q;
    const float* rstd;   // [M, H, 2]: the forward's 1/sqrt(mean(x^2)+eps) of q and k
    const float* wq;     // [128] norm weights of q and k
    const float* wk;
    const float* cosv;   // [M, 64] RoPE tables
    const float* sinv;
    uint16_t* dmixed;    // optional bf16 d(mixed_qkv) [M, 3*H*128]
    int32_t H;
    int32_t span;           // tiles per unit of work (consecutive tiles of one 128-row block)
    int32_t units_per_row;  // ceil(tiles_k / span)
    int32_t units;          // tiles_m * units_per_row
};
size_t quantize_norm_rope_smem_bytes();
int quantize_norm_rope_ctas_per_sm();
cudaError_t launch_quantize_norm_rope(const NormRopeArgs& a, int grid, cudaStream_t stream);

// Shared memory one quantizer CTA needs, and how many CTAs share an SM.
size_t quantize_smem_bytes();
int quantize_ctas_per_sm(bool sr);

// sr: elements stochastically rounded (dual only), with each task's seed.
cudaError_t launch_quantize(const QuantBatch& b, bool dual, bool sr, int grid, cudaStream_t stream);

// ---- GEMM ------------------------------------------------------------------------------
struct GemmArgs {
    int64_t M, N;        // output shape
    int32_t tiles_m;     // ceil(M / 128)
    int32_t tiles_n;     // ceil(N / 256)
    int32_t tiles_m2;    // ceil(M / 256): row tiles of the CTA-pair kernel
    int32_t group_m;     // pair kernel: row tiles per group of its tile order (1..tiles_m2)
    int32_t k_stages;    // ceil(Kp / 256): 256-element (128-byte) K steps
    int32_t kb4;         // Kp / 128: 4-block scale groups per row (scale atoms along K)
    int32_t groups_b;    // ceil(N / 128): 128-row scale groups of B
    const uint8_t* a_s;  // A scales, tensor-core layout
    const uint8_t* b_s;  // B scales, tensor-core layout
    void* c;
    int64_t ldc;
    int32_t out_f32;     // 1: fp32 output, 0: bf16
    int32_t c_tma;       // 1: cmap describes C (TMA stores), 0: plain stores
    const uint16_t* bias;  // bf16 bias[N] added to every row (16-byte aligned), or null
    uint32_t* err;
    // Output quantization (pair kernel, bf16 output through TMA stores): the MXFP4 blobs
    // of C, scales in the tensor-core layout; qo_col null: row blob only.
    uint8_t* qo_row;     // [M, Np/2]
    uint8_t* so_row;     // scales of the row blob, (M, N)
    uint8_t* qo_col;     // [N, Mp/2]
    uint8_t* so_col;     // scales of the col blob, (N, M)
    int64_t ldqo_row;    // Np / 2
    int64_t ldqo_col;    // Mp / 2
    int32_t kb4o_row;    // Np / 128: scale atoms along N
    int32_t kb4o_col;    // Mp / 128: scale atoms along M
};

size_t gemm_smem_bytes();
constexpr int kGemmBM = 128;
constexpr int kGemmBN = 256;

// amap / bmap: the element blobs as 2-D u8 tensors {Kp/2, rows}, box {128, 128 | 256},
// 128-byte swizzle, out-of-bounds bytes read as zero.  cmap (used when g.c_tma): C as a
// 2-D {N, M} tensor of its output type, box {64 bytes of columns, 32 rows}, 64-byte swizzle.
cudaError_t launch_gemm(const CUtensorMap& amap, const CUtensorMap& bmap, const CUtensorMap& cmap,
                        const GemmArgs& g, int grid, cudaStream_t stream);

// The CTA-pair kernel (gemm_pair.cu): 256 x 256 (narrow) or 256 x 384 (wide) tiles on
// clusters of two CTAs, over up to kMaxGemmTasks independent problems in one launch (tile t
// belongs to the first problem j with t < tile_end[j]; GemmArgs::tiles_n counts the
// launch's tile width).  Per problem: amap / bmap as for launch_gemm but with a B box of
// 128 rows; bmap2 (wide only): B with a box of 64 rows; sfamap / sfbmap: the A / B scale
// blobs as 2-D u64 tensors {Kp/128 * 64, ceil(rows/128)} (one row per 128-row group of
// atoms), boxes {128, 1} / {128, 2 | 3 (wide)}; cmap as for launch_gemm.  `clusters` CTA
// pairs.
constexpr int kMaxGemmTasks = 4;
struct GemmPairBatch {
    CUtensorMap amap[kMaxGemmTasks];
    CUtensorMap bmap[kMaxGemmTasks];
    CUtensorMap bmap2[kMaxGemmTasks];
    CUtensorMap cmap[kMaxGemmTasks];
    CUtensorMap sfamap[kMaxGemmTasks];
    CUtensorMap sfbmap[kMaxGemmTasks];
    GemmArgs args[kMaxGemmTasks];
    int32_t tile_end[kMaxGemmTasks];
    int32_t count;
    // Output quantization of problem 0: its row blob as a 2-D u8 tensor {Np/2, M}, box
    // {64, 32}, 64-byte swizzle; its col blob {Mp/2, N}, box {16, 128}, no swizzle.
    CUtensorMap qrowmap;
    CUtensorMap qcolmap;
};
constexpr int kPairTileNWide = 384;
size_t gemm_pair_smem_bytes(bool wide);
int gemm_pair_max_clusters(bool wide);   // co-resident clusters of the pair kernel, 0 if none
// quant: one problem (b.count == 1) whose epilogue also writes the MXFP4 blobs of C
// (GemmArgs::qo_row ..); C in bf16 through TMA stores (c_tma); narrow tiles.
// wide: 256 x 384 tiles; every problem bf16 out through TMA stores (c_tma).
cudaError_t launch_gemm_pair(const GemmPairBatch& b, int clusters, cudaStream_t stream, bool quant, bool wide);

// ---- diagnostics -----------------------------------------------------------------------
cudaError_t launch_selftest_wait(uint32_t* err, uint64_t timeout_ns, cudaStream_t stream);

}  // namespace mxfp4
