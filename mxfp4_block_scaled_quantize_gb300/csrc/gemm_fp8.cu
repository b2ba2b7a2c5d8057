// gemm_fp8.cu -- the FP8 (E5M2 x E5M2) GEMMs of the hybrid backward, on CTA pairs.
//
// `MXFP4LinearFunction.backward` in primus_turbo_mxfp4_local.py, with `backward_is_fp8`,
// computes dX = dY . W and dW = dY^T . X with `gemm_fp8_impl` on tensorwise-quantized
// E5M2 operands (TENSORWISE granularity): C = (A . B) * a_scale_inv * b_scale_inv.  With
// the column copies the quantizer writes, both are C = A . B^T over K-major operands
// (dgrad: A = dY, B = W^T; wgrad: A = dY^T, B = X^T), the form of the MXFP4 kernel.
//
// Structure as gemm_pair.cu (two CTAs on neighbouring SMs, one 256 x 256 x 32
// tcgen05.mma.kind::f8f6f4 from the even CTA reading both CTAs' shared memory; TMA
// producer in both CTAs, MMA issuer and a waiter warp in the leader, 8 epilogue warps in
// both), without scale factors.  With no scale slots, TMEM holds two 256-column
// accumulators, so tile l + 1 accumulates into the other buffer while the epilogue reads
// tile l out: the tensor pipe does not wait for the read-out at tile boundaries.  The
// epilogue multiplies by the product of the two inverse scales (read from device memory,
// where the quantizer left them) before the usual conversion and TMA store.
// Every mbarrier wait is bounded; on a timeout the CTA stops its loops, and both CTAs
// still meet at the final cluster barrier.
#include <cuda_bf16.h>

#include "epilogue.cuh"
#include "launch_fp8.h"
#include "ptx.cuh"

namespace mxfp4 {
namespace {

constexpr int BKB = 128;                  // bytes (= E5M2 elements) of K per stage
constexpr int kStages = 5;
constexpr int kABytes = 128 * BKB;        // this CTA's 128 A rows
constexpr int kBBytes = 128 * BKB;        // this CTA's 128 of the tile's 256 B rows
constexpr uint32_t kStageBytes = kABytes + kBBytes;
constexpr int kEpiWarps = 8;
constexpr int kEpi0 = 3;
constexpr int kGroupM = 8;                // row tiles per group of the tile order
constexpr int kThreads = (kEpi0 + kEpiWarps) * 32;
constexpr uint32_t kBarHandoff = 1;
constexpr uint32_t kBarEpilogue = 2;
constexpr uint32_t kAccCols = 256;
constexpr uint32_t kTmemCols = 2 * kAccCols;   // two accumulators
constexpr int kOutRowBytes = 64;
constexpr int kOutBytes = 32 * kOutRowBytes;

// Output tile lt of a problem, in groups of kGroupM 256-row tiles: within a group the row
// tile runs fastest and the groups follow each other, so the CTA pairs at work at one time
// share a few A row tiles and the B tiles of the group, which stay in L2 (row-fastest over
// the whole problem made every wave stream all of A again).
__device__ __forceinline__ void tile_coords(int lt, int tiles_m2, int tiles_n, int* mt2, int* nt) {
    const int per_group = kGroupM * tiles_n;
    const int grp = lt / per_group;
    const int first = grp * kGroupM;
    const int gm = min(tiles_m2 - first, kGroupM);
    const int r = lt - grp * per_group;
    *mt2 = first + r % gm;
    *nt = r / gm;
}

struct Fp8Smem {
    uint8_t a[kStages][kABytes];          // 1024-byte aligned (128-byte swizzle atoms)
    uint8_t b[kStages][kBBytes];
    uint8_t out[kEpiWarps][kOutBytes];
    uint64_t full[kStages];               // used in the leader: both CTAs' bytes
    uint64_t empty[kStages];              // each CTA: the leader's MMA commit
    uint64_t tmem_full[2];                // each CTA: the leader's commit after a tile
    uint64_t tmem_empty[2];               // used in the leader: 2 x kEpiWarps arrivals
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

// tcgen05.mma kind::f8f6f4: fp32 accumulator, A and B E5M2, both K-major, M = 256 (the
// pair), N = 256.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((256u >> 3) << 17) | ((256u >> 4) << 24);

__device__ __forceinline__ void tc_mma_f8_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                               uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

__device__ __forceinline__ uint32_t swz64(uint32_t r, uint32_t j) {
    return r * kOutRowBytes + ((j ^ ((r >> 1) & 3u)) << 4);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    gemm_fp8_pair_kernel(const __grid_constant__ Fp8GemmBatch P) {
    extern __shared__ uint8_t smem_raw[];
    Fp8Smem& sm = *reinterpret_cast<Fp8Smem*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const uint32_t lane = lane_id();
    const uint32_t rank = cluster_cta_rank();
    const bool leader = rank == 0;
    const int cluster = blockIdx.x >> 1;
    const int nclusters = gridDim.x >> 1;
    const int num_tiles = P.tile_end[P.count - 1];
    uint32_t* const err = P.args[0].err;
    auto task_of = [&](int t, int* local) {
        int j = 0;
        while (j + 1 < P.count && t >= P.tile_end[j]) ++j;
        *local = t - (j > 0 ? P.tile_end[j - 1] : 0);
        return j;
    };

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_addr(&sm.full[s]), 1);
            mbar_init(smem_addr(&sm.empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_addr(&sm.tmem_full[b]), 1);
            mbar_init(smem_addr(&sm.tmem_empty[b]), 2 * kEpiWarps);
        }
        mbar_init(smem_addr(&sm.drain), 1);
        sm.abort = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_addr(&sm.tmem_base), kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before_sync();
    __syncthreads();
    cluster_sync_all();
    tc_fence_after_sync();
    const uint32_t tmem = sm.tmem_base;
    grid_launch_dependents();
    grid_wait_prerequisites();

    if (warp == 0) {
        // ------------------------------------------------------------------ producer
        if (lane == 0) {
            for (int j = 0; j < P.count; ++j) {
                prefetch_tensormap(&P.amap[j]);
                prefetch_tensormap(&P.bmap[j]);
            }
            const uint64_t pol = l2_policy_evict_last();
            int it = 0;
            bool ok = true;
            for (int t = cluster; t < num_tiles && ok; t += nclusters) {
                int lt;
                const int j = task_of(t, &lt);
                const Fp8GemmArgs& g = P.args[j];
                int mt2, nt;
                tile_coords(lt, g.tiles_m2, g.tiles_n, &mt2, &nt);
                const int arow = mt2 * 256 + static_cast<int>(rank) * 128;
                const int brow = nt * 256 + static_cast<int>(rank) * 128;
                for (int ks = 0; ks < g.k_stages; ++ks, ++it) {
                    const int s = it % kStages;
                    const uint32_t ph = (it / kStages) & 1;
                    if (!mbar_wait(smem_addr(&sm.empty[s]), ph ^ 1, g.err, kErrGemmProducer, &sm.abort)) {
                        ok = false;
                        break;
                    }
                    if (leader) mbar_arrive_expect_tx(smem_addr(&sm.full[s]), 2 * kStageBytes);
                    const uint32_t bar = cluster_map(smem_addr(&sm.full[s]), 0);
                    tma_load_2d_pair(smem_addr(sm.a[s]), &P.amap[j], ks * BKB, arow, bar, pol);
                    tma_load_2d_pair(smem_addr(sm.b[s]), &P.bmap[j], ks * BKB, brow, bar, pol);
                }
            }
            if (leader) {
                const int armed = it < kStages ? it : kStages;
                for (int i = 1; i <= armed; ++i) {
                    const int j = it - i;
                    mbar_wait_quiet(smem_addr(&sm.full[j % kStages]), (j / kStages) & 1, kWaitLimitNs);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ MMA issuer
        if (leader) {
            int it = 0, tl = 0;
            bool ok = true;
            for (int t = cluster; t < num_tiles && ok; t += nclusters, ++tl) {
                int lt;
                const Fp8GemmArgs& g = P.args[task_of(t, &lt)];
                const uint32_t acc = tmem + (tl & 1) * kAccCols;
                for (int ks = 0; ks < g.k_stages; ++ks, ++it) {
                    if (!named_barrier_and(kBarHandoff, 64, true)) {
                        ok = false;
                        break;
                    }
                    if (elect_one()) {
                        tc_fence_after_sync();
                        const int s = it % kStages;
                        const uint64_t adesc = smem_desc(smem_addr(sm.a[s]), 16, 1024, 2);
                        const uint64_t bdesc = smem_desc(smem_addr(sm.b[s]), 16, 1024, 2);
#pragma unroll
                        for (int j = 0; j < BKB / 32; ++j)
                            tc_mma_f8_pair(acc, adesc + 2 * j, bdesc + 2 * j, kIdesc, (ks | j) != 0);
                        tc_commit_pair_multicast(smem_addr(&sm.empty[s]), 3);
                        if (ks == g.k_stages - 1) tc_commit_pair_multicast(smem_addr(&sm.tmem_full[tl & 1]), 3);
                    }
                    __syncwarp();
                }
            }
            if (elect_one()) {
                tc_commit_pair_multicast(smem_addr(&sm.drain), 1);
                if (!mbar_wait_quiet(smem_addr(&sm.drain), 0, kWaitLimitNs)) atomicOr(err, kErrGemmDrain);
            }
            __syncwarp();
        }
    } else if (warp == 2) {
        // ------------------------------------------------------------------ MMA waiter
        if (leader) {
            int it = 0, tl = 0;
            bool ok = true;
            for (int t = cluster; t < num_tiles && ok; t += nclusters, ++tl) {
                int lt;
                const Fp8GemmArgs& g = P.args[task_of(t, &lt)];
                for (int ks = 0; ks < g.k_stages; ++ks, ++it) {
                    int w = 1;
                    if (lane == 0) {
                        // buffer tl & 1 was last used by tile tl - 2: its read-out is the
                        // ((tl >> 1) - 1)-th completion of that buffer's tmem_empty
                        if (ks == 0 && tl >= 2)
                            w = mbar_wait(smem_addr(&sm.tmem_empty[tl & 1]), ((tl >> 1) - 1) & 1, g.err, kErrGemmMma,
                                          &sm.abort);
                        if (w)
                            w = mbar_wait(smem_addr(&sm.full[it % kStages]), (it / kStages) & 1, g.err,
                                          kErrGemmMma, &sm.abort);
                    }
                    if (!named_barrier_and(kBarHandoff, 64, __shfl_sync(0xFFFFFFFFu, w, 0) != 0)) {
                        ok = false;
                        break;
                    }
                }
            }
        }
    } else {
        // ------------------------------------------------------------------ epilogue
        const int q = warp & 3;
        const int h = (warp - kEpi0) >> 2;
        const uint32_t obuf = smem_addr(sm.out[warp - kEpi0]);
        const uint64_t pol = l2_policy_evict_first();
        const uint32_t leader_tmem_empty = cluster_map(smem_addr(&sm.tmem_empty[0]), 0);
        if (lane == 0)
            for (int j = 0; j < P.count; ++j)
                if (P.args[j].c_tma) prefetch_tensormap(&P.cmap[j]);
        int tl = 0;
        for (int t = cluster; t < num_tiles; t += nclusters, ++tl) {
            const uint32_t b = static_cast<uint32_t>(tl & 1);
            int okw = 1;
            if (warp == kEpi0 && lane == 0)
                okw = mbar_wait(smem_addr(&sm.tmem_full[b]), (tl >> 1) & 1, err, kErrGemmEpilogue, &sm.abort);
            if (!named_barrier_and(kBarEpilogue, kEpiWarps * 32, __shfl_sync(0xFFFFFFFFu, okw, 0) != 0)) break;
            tc_fence_after_sync();
            uint32_t v[4][32];
            const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + b * kAccCols + h * 128;
            tc_ld_32x32b_x32(taddr + 0, v[0]);
            tc_ld_32x32b_x32(taddr + 32, v[1]);
            tc_ld_32x32b_x32(taddr + 64, v[2]);
            tc_ld_32x32b_x32(taddr + 96, v[3]);
            tc_wait_ld();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster_relaxed(leader_tmem_empty + b * 8u);

            int lt;
            const int pj = task_of(t, &lt);
            const Fp8GemmArgs& g = P.args[pj];
            int mt2, nt;
            tile_coords(lt, g.tiles_m2, g.tiles_n, &mt2, &nt);
            const int64_t row0 = static_cast<int64_t>(mt2) * 256 + rank * 128 + q * 32;
            const int64_t col0 = static_cast<int64_t>(nt) * 256 + h * 128;
            if (row0 >= g.M || col0 >= g.N) continue;
            // the two tensors' inverse scales, multiplied in fp32
            const float s = __fmul_rn(__ldg(g.a_scale_inv), __ldg(g.b_scale_inv));
#pragma unroll
            for (int c4 = 0; c4 < 4; ++c4)
#pragma unroll
                for (int i = 0; i < 32; ++i) v[c4][i] = __float_as_uint(__fmul_rn(__uint_as_float(v[c4][i]), s));
            if (g.c_tma) {
                const int per = g.out_f32 ? 16 : 32;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    if (c * per >= 128 || col0 + c * per >= g.N) break;
                    if (lane == 0) bulk_wait_read_all();
                    __syncwarp();
                    uint32_t w[16];
                    if (g.out_f32)
                        convert_piece<true>(&v[(c >> 1) & 3][(c & 1) * 16], nullptr, col0 + c * per, g.N, w);
                    else
                        convert_piece<false>(v[c & 3], nullptr, col0 + c * per, g.N, w);
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        sts128(obuf + swz64(lane, j), w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d_hint(&P.cmap[pj], static_cast<int32_t>(col0 + c * per), static_cast<int32_t>(row0),
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
                        if (col0 + c4 * 32 + j < g.N) dst[c4 * 32 + j] = out_bf16(v[c4][j], nullptr, 0);
            } else {
                float* dst = reinterpret_cast<float*>(g.c) + row * g.ldc + col0;
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4)
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (col0 + c4 * 32 + j < g.N) dst[c4 * 32 + j] = out_f32(v[c4][j], nullptr, 0);
            }
        }
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    }

    tc_fence_before_sync();
    __syncthreads();
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc_pair(tmem, kTmemCols);
    }
}

}  // namespace

size_t gemm_fp8_smem_bytes() { return sizeof(Fp8Smem) + 1024; }

int gemm_fp8_max_clusters() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cached[dev] > 0) return cached[dev];
    const size_t smem = gemm_fp8_smem_bytes();
    if (cudaFuncSetAttribute(gemm_fp8_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
        cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_fp8_pair_kernel, &cfg) != cudaSuccess) return 0;
    cached[dev] = n;
    return n;
}

cudaError_t launch_gemm_fp8(const Fp8GemmBatch& b, int clusters, cudaStream_t stream) {
    const size_t smem = gemm_fp8_smem_bytes();
    cudaError_t e = cudaFuncSetAttribute(gemm_fp8_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * clusters, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemm_fp8_pair_kernel, b);
}

}  // namespace mxfp4
