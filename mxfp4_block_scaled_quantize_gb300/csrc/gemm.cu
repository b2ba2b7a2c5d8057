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
//               into a 4-stage shared-memory ring.  Operands are read with an L2
//               evict-last policy: every tile row and column is read many times.
//   warp 1      allocates TMEM (512 columns: accumulator in 0..255, per-stage scale slots
//               after it).  The whole warp walks the schedule and one elected lane issues,
//               per stage, the six scale copies (tcgen05.cp) and four 128x256x64
//               block-scaled MMAs, then commits the stage back to the producer and, after
//               a tile's last K step, the accumulator to the epilogue.  This warp never
//               waits on a shared-memory barrier and never branches around its tensor
//               instructions: on this part either one holds each copy back until the MMAs
//               queued before it are done, which costs about 80% of the MMA rate.  So
//   warp 2      waits on the barriers for it and hands each stage over through a named
//               barrier whose AND-reduction also carries the ok / give-up flag.
//   warps 3..10 epilogue: each warp owns one 32-lane quadrant and one 128-column half of
//               the accumulator.  It pulls its 32 x 128 fp32 values into registers, frees
//               the accumulator at once (so the next tile's MMAs overlap the stores),
//               converts them and writes them out through a 2 KB swizzled shared-memory
//               buffer with TMA stores (L2 evict-first: C is written once), which keeps
//               the load/store unit free for the barrier traffic of warps 0 and 2.  A C
//               whose pitch breaks the TMA rules is written with plain stores.
// Every wait is bounded (see ptx.cuh); a wait that runs out stops the CTA cleanly.
#include <cuda_bf16.h>

#include "epilogue.cuh"
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
constexpr int kEpi0 = 3;                  // warps 0 producer, 1 MMA, 2 MMA waiter
constexpr int kThreads = (kEpi0 + kEpiWarps) * 32;
constexpr uint32_t kBarHandoff = 1;       // named barrier: MMA warp + waiter warp
constexpr uint32_t kBarEpilogue = 2;      // named barrier: the epilogue warps
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSfTmemBase = BN;      // scale slots start after the accumulator
constexpr uint32_t kSfTmemPerStage = 24;  // SFA 2 atoms x 4 cols + SFB 2 atoms x 2 groups x 4
constexpr int kOutRowBytes = 64;          // bytes of one output row per TMA store
constexpr int kOutBytes = 32 * kOutRowBytes;

struct GemmSmem {
    uint8_t a[kStages][kABytes];          // 1024-byte aligned (128-byte swizzle atoms)
    uint8_t b[kStages][kBBytes];
    uint8_t sfa[kStages][kSfaBytes];
    uint8_t sfb[kStages][kSfbBytes];
    uint8_t out[kEpiWarps][kOutBytes];    // 512-byte aligned (64-byte swizzle atoms)
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

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

// Byte offset of 16-byte chunk j (0..3) of row r in a 64-byte-swizzled box of 64-byte rows:
// the chunk index is XORed with bits 7..8 of the row's byte offset.
__device__ __forceinline__ uint32_t swz64(uint32_t r, uint32_t j) {
    return r * kOutRowBytes + ((j ^ ((r >> 1) & 3u)) << 4);
}

template <bool kBias>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_mxf4_kernel(const __grid_constant__ CUtensorMap amap, const __grid_constant__ CUtensorMap bmap,
                     const __grid_constant__ CUtensorMap cmap, const GemmArgs g) {
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
    grid_launch_dependents();
    grid_wait_prerequisites();

    if (warp == 0) {
        // ------------------------------------------------------------------ producer
        if (lane == 0) {
            prefetch_tensormap(&amap);
            prefetch_tensormap(&bmap);
            const uint64_t pol = l2_policy_evict_last();
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
                    tma_load_2d_hint(smem_addr(sm.a[s]), &amap, ks * BKB, mt * BM, bar, pol);
                    tma_load_2d_hint(smem_addr(sm.b[s]), &bmap, ks * BKB, nt * BN, bar, pol);
                    bulk_load_hint(smem_addr(sm.sfa[s]),
                                   g.a_s + (static_cast<int64_t>(mt) * g.kb4 + 2 * ks) * 512, natoms * 512,
                                   bar, pol);
                    for (int gi = 0; gi < ngroups; ++gi)
                        bulk_load_hint(smem_addr(sm.sfb[s]) + gi * 1024,
                                       g.b_s + (static_cast<int64_t>(2 * nt + gi) * g.kb4 + 2 * ks) * 512,
                                       natoms * 512, bar, pol);
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
        // All 32 lanes walk the schedule; no shared-memory access until the drain.
        int it = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
            for (int ks = 0; ks < g.k_stages; ++ks, ++it) {
                // Stage landed (and, on a tile's first step, accumulator free).
                if (!named_barrier_and(kBarHandoff, 64, true)) {
                    ok = false;
                    break;
                }
                if (elect_one()) {
                    tc_fence_after_sync();
                    const int s = it % kStages;
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
                        // MMA j: 64 elements = 32 bytes further into each swizzled row.
                        const uint32_t sf_id = (j & 1) * 2;
                        tc_mma_mxf4(tmem, adesc + 2 * j, bdesc + 2 * j, mma_idesc(sf_id),
                                    sf + (j >> 1) * 4, sf + 8 + (j >> 1) * 8, (ks | j) != 0);
                    }
                    tc_commit(smem_addr(&sm.empty[s]));
                    if (ks == g.k_stages - 1) tc_commit(smem_addr(&sm.tmem_full));
                }
            }
        }
        // Drain: all MMAs and copies issued by this warp complete before teardown.
        if (elect_one()) {
            tc_commit(smem_addr(&sm.drain));
            if (!mbar_wait_quiet(smem_addr(&sm.drain), 0, kWaitLimitNs)) atomicOr(g.err, kErrGemmDrain);
        }
        __syncwarp();
    } else if (warp == 2) {
        // ------------------------------------------------------------------ MMA waiter
        // Mirrors the MMA warp's schedule: before each hand-over, lane 0 waits for what the
        // MMA warp is about to use; the AND-reduction passes a failed wait on.
        int it = 0, tl = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x, ++tl) {
            for (int ks = 0; ks < g.k_stages; ++ks, ++it) {
                int w = 1;
                if (lane == 0) {
                    if (ks == 0 && tl > 0)
                        w = mbar_wait(smem_addr(&sm.tmem_empty), (tl - 1) & 1, g.err, kErrGemmMma, &sm.abort);
                    if (w)
                        w = mbar_wait(smem_addr(&sm.full[it % kStages]), (it / kStages) & 1, g.err, kErrGemmMma,
                                      &sm.abort);
                }
                if (!named_barrier_and(kBarHandoff, 64, __shfl_sync(0xFFFFFFFFu, w, 0) != 0)) {
                    ok = false;
                    break;
                }
            }
        }
    } else {
        // ------------------------------------------------------------------ epilogue
        const int q = warp & 3;                  // TMEM lane quadrant this warp may access
        const int h = (warp - kEpi0) >> 2;       // column half of the tile
        const uint32_t obuf = smem_addr(sm.out[warp - kEpi0]);
        const uint64_t pol = l2_policy_evict_first();
        if (g.c_tma && lane == 0) prefetch_tensormap(&cmap);
        int tl = 0;
        for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++tl) {
            // One lane polls the accumulator barrier; the other warps sleep on a named one.
            int okw = 1;
            if (warp == kEpi0 && lane == 0)
                okw = mbar_wait(smem_addr(&sm.tmem_full), tl & 1, g.err, kErrGemmEpilogue, &sm.abort);
            if (!named_barrier_and(kBarEpilogue, kEpiWarps * 32, __shfl_sync(0xFFFFFFFFu, okw, 0) != 0)) break;
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
            if (lane == 0) mbar_arrive_relaxed(smem_addr(&sm.tmem_empty));

            const int mt = t % g.tiles_m, nt = t / g.tiles_m;
            const int64_t row0 = static_cast<int64_t>(mt) * BM + q * 32;
            const int64_t col0 = static_cast<int64_t>(nt) * BN + h * 128;
            if (row0 >= g.M || col0 >= g.N) continue;
            if (g.c_tma) {
                // 64-byte row pieces: 32 bf16 or 16 fp32 columns per store; the tensor map
                // leaves rows >= M and columns >= N unwritten.
                const int per = g.out_f32 ? 16 : 32;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    if (c * per >= 128 || col0 + c * per >= g.N) break;
                    if (lane == 0) bulk_wait_read_all();   // the buffer's previous store has read it
                    __syncwarp();
                    uint32_t w[16];
                    const uint16_t* const bias = kBias ? g.bias : nullptr;
                    if (g.out_f32)
                        convert_piece<true>(&v[(c >> 1) & 3][(c & 1) * 16], bias, col0 + c * per, g.N, w);
                    else
                        convert_piece<false>(v[c & 3], bias, col0 + c * per, g.N, w);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        sts128(obuf + swz64(lane, j), w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d_hint(&cmap, static_cast<int32_t>(col0 + c * per), static_cast<int32_t>(row0),
                                          obuf, pol);
                        bulk_commit_group();
                    }
                }
                continue;
            }
            const int64_t row = row0 + lane;
            if (row >= g.M) continue;
            if (!g.out_f32) {
                __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(g.c) + row * g.ldc + col0;
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4)
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (col0 + c4 * 32 + j < g.N) dst[c4 * 32 + j] = out_bf16(v[c4][j], kBias ? g.bias : nullptr, col0 + c4 * 32 + j);
            } else {
                float* dst = reinterpret_cast<float*>(g.c) + row * g.ldc + col0;
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4)
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (col0 + c4 * 32 + j < g.N) dst[c4 * 32 + j] = out_f32(v[c4][j], kBias ? g.bias : nullptr, col0 + c4 * 32 + j);
            }
        }
        // Every TMA store of this warp is complete before the CTA may leave.
        if (lane == 0) bulk_wait_all();
        __syncwarp();
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

cudaError_t launch_gemm(const CUtensorMap& amap, const CUtensorMap& bmap, const CUtensorMap& cmap,
                        const GemmArgs& g, int grid, cudaStream_t stream) {
    const size_t smem = gemm_smem_bytes();
    auto kernel = g.bias != nullptr ? gemm_mxf4_kernel<true> : gemm_mxf4_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, amap, bmap, cmap, g);
}

}  // namespace mxfp4
