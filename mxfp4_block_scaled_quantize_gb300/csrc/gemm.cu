// gemm.cu -- block-scaled MXF4 GEMM on the sm_103a tensor cores (tcgen05, kind::mxf4).
//
// C[M,N] = A[M,K] . B[N,K]^T where A and B are K-packed MXFP4 blobs (FP4 E2M1 elements,
// one E8M0 scale per 32 elements, scales in the tensor-core layout).  This is the one
// GEMM form the forward (Y = X.W^T: A = X row blob, B = W row blob), dgrad
// (dX = dY.W: A = dY row blob, B = W col blob) and wgrad (dW = dY^T.X: A = dY col blob,
// B = X col blob) calls of `MXFP4LinearFunction` in primus_turbo_mxfp4_local.py take.
// Products accumulate in fp32 in tensor memory; the output is fp32 or bf16 (rounded
// once, to nearest even).
//
// Design (one CTA per SM, persistent over 128 x 256 output tiles, warp-specialized):
//   warp 0      one thread issues TMA: per 256-element K step, the A tile (128 rows x 128
//               bytes) and B tile (256 x 128 bytes) with 128-byte swizzle, and the scale
//               atoms of both (512 bytes per 128 rows x 128 K) with plain bulk copies,
//               into a 4-stage shared-memory ring.
//   warp 1      allocates TMEM (512 columns: accumulator in 0..255, per-stage scale slots
//               after it); one thread copies each stage's scales to TMEM (tcgen05.cp) and
//               issues four 128x256x64 block-scaled MMAs per stage, then commits the stage
//               back to the producer and, after the last K step, the tile to the epilogue.
//   warps 2..9  epilogue: each warp owns one 32-lane quadrant and one 128-column half of
//               the accumulator; it pulls its 32 x 128 fp32 values into registers, frees
//               the accumulator at once (so the next tile's MMAs overlap the stores), then
//               converts and stores them.
// Every wait is bounded (see ptx.cuh); a wait that runs out stops the CTA cleanly.
#include <cuda_bf16.h>

#include "launch.h"
#include "ptx.cuh"

namespace mxfp4 {
namespace {

constexpr int BM = kGemmBM;               // 128 output rows per tile
constexpr int BN = kGemmBN;               // 256 output columns per tile
constexpr int BKB = 128;                  // bytes of K per stage (256 FP4 elements)
constexpr int kStages = 4;
constexpr int kABytes = BM * BKB;         // 16 KB
constexpr int kBBytes = BN * BKB;         // 32 KB
constexpr int kSfaBytes = 2 * 512;        // 2 scale atoms (K 256) for 128 rows
constexpr int kSfbBytes = 2 * 2 * 512;    // 2 row groups x 2 atoms
constexpr int kEpiWarps = 8;
constexpr int kThreads = (2 + kEpiWarps) * 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfTmemBase = BN;      // scale slots start after the accumulator
constexpr uint32_t kSfTmemPerStage = 24;  // SFA 2 atoms x 4 cols + SFB 2 atoms x 2 groups x 4

struct GemmSmem {
    uint8_t a[kStages][kABytes];          // 1024-byte aligned (128-byte swizzle atoms)
    uint8_t b[kStages][kBBytes];
    uint8_t sfa[kStages][kSfaBytes];
    uint8_t sfb[kStages][kSfbBytes];
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t tmem_full;
    uint64_t tmem_empty;
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

// Instruction descriptor of tcgen05.mma kind::mxf4: E2M1 A and B, K-major both, fp32
// accumulate, E8M0 scales, M = 128, N = 256; scale-factor byte selectors sfa_id / sfb_id.
__device__ __forceinline__ uint32_t mma_idesc(uint32_t sf_id) {
    uint32_t d = 0;
    d |= sf_id << 4;                          // B scale-factor byte selector
    d |= 1u << 7;                             // A format: E2M1
    d |= 1u << 10;                            // B format: E2M1
    d |= static_cast<uint32_t>(BN >> 3) << 17;
    d |= 1u << 23;                            // scale format: UE8M0
    d |= static_cast<uint32_t>(BM >> 4) << 24;
    d |= sf_id << 29;                         // A scale-factor byte selector
    return d;
}

__device__ __forceinline__ uint32_t pack_bf16x2(uint32_t lo_bits, uint32_t hi_bits) {
    __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(lo_bits), __uint_as_float(hi_bits));
    return *reinterpret_cast<uint32_t*>(&h);
}

__global__ void __launch_bounds__(kThreads, 1)
    gemm_mxf4_kernel(const __grid_constant__ CUtensorMap amap, const __grid_constant__ CUtensorMap bmap,
                     const GemmArgs g) {
    extern __shared__ uint8_t smem_raw[];
    GemmSmem& sm = *reinterpret_cast<GemmSmem*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const uint32_t lane = lane_id();
    const int num_tiles = g.tiles_m * g.tiles_n;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_addr(&sm.full[s]), 1);
            mbar_init(smem_addr(&sm.empty[s]), 1);
        }
        mbar_init(smem_addr(&sm.tmem_full), 1);
        mbar_init(smem_addr(&sm.tmem_empty), kEpiWarps);
        mbar_init(smem_addr(&sm.drain), 1);
        sm.abort = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(&sm.tmem_base), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = sm.tmem_base;

    if (warp == 0) {
        // ------------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tensormap(&amap);
            prefetch_tensormap(&bmap);
            int it = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
                const int mt = t % g.tiles_m, nt = t / g.tiles_m;
                const int ngroups = min(2, g.groups_b - 2 * nt);
                for (int ks = 0; ks < g.k_stages; ++ks, ++it) {
                    const int s = it % kStages;
                    const uint32_t ph = (it / kStages) & 1;
                    if (!mbar_wait(smem_addr(&sm.empty[s]), ph ^ 1, g.err, kErrGemmProducer, &sm.abort)) {
                        ok = false;
                        break;
                    }
                    const int natoms = min(2, g.kb4 - 2 * ks);
                    const uint32_t bar = smem_addr(&sm.full[s]);
                    mbar_arrive_expect_tx(bar, kABytes + kBBytes + natoms * 512 * (1 + ngroups));
                    tma_load_2d(smem_addr(sm.a[s]), &amap, ks * BKB, mt * BM, bar);
                    tma_load_2d(smem_addr(sm.b[s]), &bmap, ks * BKB, nt * BN, bar);
                    bulk_load(smem_addr(sm.sfa[s]),
                              g.a_s + (static_cast<int64_t>(mt) * g.kb4 + 2 * ks) * 512, natoms * 512, bar);
                    for (int gi = 0; gi < ngroups; ++gi)
                        bulk_load(smem_addr(sm.sfb[s]) + gi * 1024,
                                  g.b_s + (static_cast<int64_t>(2 * nt + gi) * g.kb4 + 2 * ks) * 512,
                                  natoms * 512, bar);
                }
            }
            // Drain: every armed stage's copies have landed before this thread may leave.
            const int armed = it < kStages ? it : kStages;
            for (int i = 1; i <= armed; ++i) {
                const int j = it - i;
                mbar_wait_quiet(smem_addr(&sm.full[j % kStages]), (j / kStages) & 1, kWaitLimitNs);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int it = 0, tl = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x, ++tl) {
                if (tl > 0) {
                    if (!mbar_wait(smem_addr(&sm.tmem_empty), (tl - 1) & 1, g.err, kErrGemmMma, &sm.abort))
                        break;
                    tc_fence_after_sync();
                }
                for (int ks = 0; ks < g.k_stages; ++ks, ++it) {
                    const int s = it % kStages;
                    const uint32_t ph = (it / kStages) & 1;
                    if (!mbar_wait(smem_addr(&sm.full[s]), ph, g.err, kErrGemmMma, &sm.abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const int natoms = min(2, g.kb4 - 2 * ks);
                    const uint32_t sf = tmem + kSfTmemBase + s * kSfTmemPerStage;
                    const uint32_t sfa_s = smem_addr(sm.sfa[s]);
                    const uint32_t sfb_s = smem_addr(sm.sfb[s]);
                    // Scale atoms: 32 lines x 16 bytes, 8-line core groups 128 bytes apart.
                    for (int a = 0; a < natoms; ++a) {
                        tc_cp_32x128b_warpx4(sf + a * 4, smem_desc(sfa_s + a * 512, 0, 128, 0));
                        tc_cp_32x128b_warpx4(sf + 8 + a * 8, smem_desc(sfb_s + a * 512, 0, 128, 0));
                        tc_cp_32x128b_warpx4(sf + 8 + a * 8 + 4, smem_desc(sfb_s + 1024 + a * 512, 0, 128, 0));
                    }
                    const uint64_t adesc = smem_desc(smem_addr(sm.a[s]), 16, 1024, 2);
                    const uint64_t bdesc = smem_desc(smem_addr(sm.b[s]), 16, 1024, 2);
                    for (int j = 0; j < natoms * 2; ++j) {
                        // K step j: 64 elements = 32 bytes further into each swizzled row.
                        const uint32_t sf_id = (j & 1) * 2;
                        tc_mma_mxf4(tmem, adesc + 2 * j, bdesc + 2 * j, mma_idesc(sf_id),
                                    sf + (j >> 1) * 4, sf + 8 + (j >> 1) * 8, (ks | j) != 0);
                    }
                    tc_commit(smem_addr(&sm.empty[s]));
                }
                if (!ok) break;
                tc_commit(smem_addr(&sm.tmem_full));
            }
            // Drain: all MMAs and copies issued by this thread complete before teardown.
            tc_commit(smem_addr(&sm.drain));
            if (!mbar_wait_quiet(smem_addr(&sm.drain), 0, kWaitLimitNs)) atomicOr(g.err, kErrGemmDrain);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------------ epilogue
        const int q = warp & 3;                  // TMEM lane quadrant this warp may access
        const int h = (warp - 2) >> 2;           // column half of the tile
        int tl = 0;
        for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++tl) {
            int okw = 0;
            if (lane == 0)
                okw = mbar_wait(smem_addr(&sm.tmem_full), tl & 1, g.err, kErrGemmEpilogue, &sm.abort);
            okw = __shfl_sync(0xFFFFFFFFu, okw, 0);
            if (!okw) break;
            tc_fence_after_sync();
            uint32_t v[4][32];
            const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + h * 128;
            tc_ld_32x32b_x32(taddr + 0, v[0]);
            tc_ld_32x32b_x32(taddr + 32, v[1]);
            tc_ld_32x32b_x32(taddr + 64, v[2]);
            tc_ld_32x32b_x32(taddr + 96, v[3]);
            tc_wait_ld();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&sm.tmem_empty));

            const int mt = t % g.tiles_m, nt = t / g.tiles_m;
            const int64_t row = static_cast<int64_t>(mt) * BM + q * 32 + lane;
            const int64_t col0 = static_cast<int64_t>(nt) * BN + h * 128;
            if (row >= g.M) continue;
            const bool full_cols = col0 + 128 <= g.N;
            if (!g.out_f32) {
                __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(g.c) + row * g.ldc + col0;
                if (full_cols && (g.ldc & 7) == 0) {
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4)
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const uint32_t* x = &v[c4][8 * j];
                            uint4 pk = make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]),
                                                  pack_bf16x2(x[4], x[5]), pack_bf16x2(x[6], x[7]));
                            *reinterpret_cast<uint4*>(dst + c4 * 32 + 8 * j) = pk;
                        }
                } else {
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4)
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (col0 + c4 * 32 + j < g.N)
                                dst[c4 * 32 + j] = __float2bfloat16_rn(__uint_as_float(v[c4][j]));
                }
            } else {
                float* dst = reinterpret_cast<float*>(g.c) + row * g.ldc + col0;
                if (full_cols && (g.ldc & 3) == 0) {
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4)
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            *reinterpret_cast<uint4*>(dst + c4 * 32 + 4 * j) =
                                make_uint4(v[c4][4 * j], v[c4][4 * j + 1], v[c4][4 * j + 2], v[c4][4 * j + 3]);
                } else {
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4)
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (col0 + c4 * 32 + j < g.N) dst[c4 * 32 + j] = __uint_as_float(v[c4][j]);
                }
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

size_t gemm_smem_bytes() { return sizeof(GemmSmem) + 1024; }

cudaError_t launch_gemm(const CUtensorMap& amap, const CUtensorMap& bmap, const GemmArgs& g, int grid,
                        cudaStream_t stream) {
    const size_t smem = gemm_smem_bytes();
    cudaError_t e = cudaFuncSetAttribute(gemm_mxf4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    gemm_mxf4_kernel<<<grid, kThreads, smem, stream>>>(amap, bmap, g);
    return cudaGetLastError();
}

}  // namespace mxfp4
