// gemm_pair.cu -- the block-scaled MXF4 GEMM on CTA pairs (tcgen05 cta_group::2).
//
// Same operation and operands as gemm.cu (C = A . B^T on K-packed MXFP4 blobs with scales
// in the tensor-core layout, fp32 accumulation, fp32 or bf16 out), for problems with more
// than one 128-row tile.  A cluster of two CTAs on neighbouring SMs owns 256 x 256 output
// tiles: each CTA holds the A rows of its own 128-row half and half of the tile's B rows,
// and one 256 x 256 x 64 MMA issued by the even CTA reads both CTAs' shared memory.  Per
// SM that is 35 KB of operands per 256-element K step instead of 51 KB for a 128 x 256
// tile on one SM, so the same shared memory holds five stages instead of four and L2
// feeds a third fewer bytes per flop.  The wide instances own 256 x 384 tiles (PairCfg).
//
// Layout facts this relies on (measured on the part: each CTA's scale copy lands in its
// own TMEM from its own shared memory, and each SM reads all N B-scales from its own TMEM):
//   - every CTA loads the A scales of its own rows and the B scales of all the tile's rows;
//   - all loads of a stage, from both CTAs, complete on the even CTA's `full` barrier;
//   - the MMA's commit arrives on `empty` / `tmem_full` in both CTAs (multicast).
//
// Roles (both CTAs run the same code; `leader` is the even CTA):
//   warp 0      producer, both CTAs: per K step, its A half (128 rows x 128 bytes), its B
//               half (128 x 128; wide: and 64 more rows), its A scales (1 KB) and all B
//               scales (2 KB; wide 3 KB) by TMA.
//   warp 1      TMEM allocation for the pair (512 columns, same address in both CTAs); in
//               the leader, the MMA issuer (one elected lane of a converged warp).
//   warp 2      leader only: waits on the barriers for the MMA warp, named-barrier hand-over.
//   warps 3..   epilogue, both CTAs (8 warps; wide 12): the CTA's own 128 accumulator
//               rows, a lane quarter x 128 columns per warp; each warp reports the
//               accumulator read to the leader's `tmem_empty`.
// Every mbarrier wait is bounded; on a timeout the CTA stops its loops, and both CTAs
// still meet at the final cluster barrier, so neither leaves while the other may touch
// its shared memory.
#include <cuda_bf16.h>

#include "epilogue.cuh"
#include "launch.h"
#include "mx_encode.cuh"
#include "ptx.cuh"

namespace mxfp4 {
namespace {

constexpr int BKB = 128;                  // bytes of K per stage (256 FP4 elements)
constexpr int kABytes = 128 * BKB;        // this CTA's 128 A rows
constexpr int kSfaBytes = 2 * 512;        // 2 scale atoms of this CTA's rows
constexpr int kEpi0 = 3;
constexpr uint32_t kBarHandoff = 1;
constexpr uint32_t kBarEpilogue = 2;
constexpr uint32_t kBarStore0 = 3;        // wide: + column group h, the group's four warps
constexpr uint32_t kTmemCols = 512;
constexpr int kOutRowBytes = 64;
constexpr int kOutBytes = 32 * kOutRowBytes;

// Tile shapes.  Narrow: 256 x 256 tiles, one N 256 MMA per K slice, five stages.  Wide:
// 256 x 384 tiles, per K slice an N 256 MMA (tile columns 0..255, accumulator columns
// 0..255) and an N 128 MMA (tile columns 256..383, accumulator columns 256..383) on the
// same A; each CTA stages B rows [128 r, 128 r + 128) and [256 + 64 r, 256 + 64 r + 64) of
// the tile (r its rank), the halves the two MMAs take from it.  Per SM that is 44 KB of
// operands for 1.5x the flops of a narrow K step (a sixth fewer bytes per flop), four stages,
// and one accumulator hand-over per 1.5x the work; the 384 accumulator columns and four
// stages of 32 scale columns fill the 512 TMEM columns.  12 epilogue warps.
template <bool kWide>
struct PairCfg {
    static constexpr int kTileN = kWide ? 384 : 256;
    static constexpr int kStages = kWide ? 4 : 5;
    static constexpr int kBRows = kWide ? 192 : 128;   // this CTA's B rows per stage
    static constexpr int kBBytes = kBRows * BKB;
    static constexpr int kBGroups = kTileN / 128;      // 128-row scale groups of the tile's B
    static constexpr int kSfbBytes = kBGroups * 2 * 512;
    static constexpr uint32_t kStageBytes = kABytes + kBBytes + kSfaBytes + kSfbBytes;
    static constexpr int kEpiWarps = kTileN / 32;      // 4 lane quarters x 128-column groups
    static constexpr int kThreads = (kEpi0 + kEpiWarps) * 32;
    static constexpr uint32_t kSfTmemBase = kTileN;    // after the accumulator
    static constexpr uint32_t kSfTmemPerStage = 4 * (2 + 2 * kBGroups);
    static constexpr int kQuantWarps = kWide ? 1 : kEpiWarps;   // output quantization: narrow only
};
static_assert(PairCfg<false>::kSfTmemBase + PairCfg<false>::kStages * PairCfg<false>::kSfTmemPerStage <= kTmemCols,
              "narrow TMEM budget");
static_assert(PairCfg<true>::kSfTmemBase + PairCfg<true>::kStages * PairCfg<true>::kSfTmemPerStage <= kTmemCols,
              "wide TMEM budget");

template <bool kWide>
struct PairSmem {
    using C = PairCfg<kWide>;
    uint8_t a[C::kStages][kABytes];       // 1024-byte aligned (128-byte swizzle atoms)
    uint8_t b[C::kStages][C::kBBytes];
    uint8_t sfa[C::kStages][kSfaBytes];
    uint8_t sfb[C::kStages][C::kSfbBytes];
    uint8_t out[C::kEpiWarps][kOutBytes];
    // output quantization: per epilogue warp, the row-blob codes of its 32 rows x 128
    // columns (32 x 64 bytes, 64-byte swizzle) and the col-blob codes of its 128 columns x 32
    // rows (128 x 16 bytes), each leaving in one tensor store
    uint8_t qrow[C::kQuantWarps][kOutBytes];
    uint8_t qcol[C::kQuantWarps][kOutBytes];
    uint64_t full[C::kStages];            // used in the leader: both CTAs' bytes
    uint64_t empty[C::kStages];           // each CTA: the leader's MMA commit
    uint64_t tmem_full;                   // each CTA: the leader's commit after a tile
    uint64_t tmem_empty;                  // used in the leader: 2 x kEpiWarps arrivals
    uint64_t drain;
    uint32_t tmem_base;
    int abort;
};

// tcgen05.mma kind::mxf4 instruction descriptor, M = 256 (the pair), N = n.
__device__ __forceinline__ uint32_t pair_idesc(uint32_t sf_id, uint32_t n) {
    uint32_t d = 0;
    d |= sf_id << 4;
    d |= 1u << 7;
    d |= 1u << 10;
    d |= (n >> 3) << 17;
    d |= 1u << 23;
    d |= static_cast<uint32_t>(256 >> 4) << 24;
    d |= sf_id << 29;
    return d;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

__device__ __forceinline__ void sts32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t swz64(uint32_t r, uint32_t j) {
    return r * kOutRowBytes + ((j ^ ((r >> 1) & 3u)) << 4);
}

// Four 8 x 8 bf16 matrices from shared memory, transposed: lanes 8j .. 8j + 7 give the
// addresses of the 8 rows (16 bytes each) of matrix j, and lane t receives in d[j] the
// elements (row 2 (t % 4), column t / 4) (low half) and (row 2 (t % 4) + 1, column t / 4).
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t* d) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
                 : "r"(addr));
}

__device__ __forceinline__ uint32_t lds_u16(uint32_t addr) {
    uint16_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
    return v;
}

// Output quantization of one staged 32 x 32 piece c of bf16 C (rows row0 .. row0 + 31 of
// the warp, columns col .. col + 31): w holds this lane's row of the piece (bf16 pairs, even
// column low), `obuf` the same piece in shared memory (swz64 layout).  Row blob: the lane's
// 32-element block, its 16 code bytes staged as chunk c of row `lane` in `qrow` (swz64
// layout), its scale byte (0 for a padding row) in byte c of *srow.  Col blob (g.qo_col
// set): column col + lane, read back down the 32 staged rows (rows past M count as 0), its
// 16 code bytes staged as row 32 c + lane of `qcol`, its scale byte written straight into
// the tensor-core layout (0 for a padding column).  The elements, scales and padding are
// those the quantizer gives for C's bf16 values; the tensor stores clip rows past M (row
// blob) and columns past N (col blob).
__device__ __forceinline__ void quantize_out_piece(const GemmArgs& g, const uint32_t* w, uint32_t obuf,
                                                   uint32_t qrow, uint32_t qcol, int64_t row0, int64_t col, int c,
                                                   int q, uint32_t lane, uint32_t* srow) {
    const int64_t row = row0 + lane;
    uint32_t m = w[0];
#pragma unroll
    for (int i = 1; i < 16; ++i) m = absmax2(m, w[i]);
    m = absmax2(m, m >> 16) & 0x7FFFu;   // even and odd columns folded: the block's amax
    const uint32_t rbyte = row < g.M ? scale_byte(m) : 0u;
    *srow |= rbyte << (8 * c);
    {
        const uint64_t s2 = pack2(inv_scale_bits(rbyte), inv_scale_bits(rbyte));
        sts128(qrow + swz64(lane, c), encode8(w[0], w[1], w[2], w[3], s2), encode8(w[4], w[5], w[6], w[7], s2),
               encode8(w[8], w[9], w[10], w[11], s2), encode8(w[12], w[13], w[14], w[15], s2));
    }
    if (g.qo_col == nullptr) return;
    const int64_t n_pad = (g.N + 127) & ~int64_t{127};
    if (row0 + 32 <= g.M) {
        // The usual case, every row of the block a row of C: four transposing matrix loads
        // give lane t the row pairs (8 rb + 2 (t % 4), + 1), rb = 0..3, of the piece's columns
        // 8 cb + t / 4, cb = 0..3.  A column's amax is folded over its four lanes, and its
        // codes -- lane t % 4 = q' holding bytes 4 rb + q' -- are transposed across those
        // lanes so that lane q' holds bytes 4 q' .. 4 q' + 3.
        uint32_t wc[4][4];   // [cb][rb]
#pragma unroll
        for (int rb = 0; rb < 4; ++rb) {
            uint32_t d[4];
            ldsm_x4_trans(obuf + swz64(8 * rb + (lane & 7u), lane >> 3), d);
#pragma unroll
            for (int cb = 0; cb < 4; ++cb) wc[cb][rb] = d[cb];
        }
        uint32_t mc[4];
#pragma unroll
        for (int cb = 0; cb < 4; ++cb) {
            const uint32_t m4 = absmax2(absmax2(wc[cb][0], wc[cb][1]), absmax2(wc[cb][2], wc[cb][3]));
            mc[cb] = absmax2(m4, m4 >> 16) & 0x7FFFu;
        }
        uint32_t p01 = mc[0] | (mc[1] << 16), p23 = mc[2] | (mc[3] << 16);
        p01 = absmax2(p01, __shfl_xor_sync(0xFFFFFFFFu, p01, 1));
        p23 = absmax2(p23, __shfl_xor_sync(0xFFFFFFFFu, p23, 1));
        p01 = absmax2(p01, __shfl_xor_sync(0xFFFFFFFFu, p01, 2));
        p23 = absmax2(p23, __shfl_xor_sync(0xFFFFFFFFu, p23, 2));
        const uint32_t qq = lane & 3u;
        const uint32_t sel_a = (qq & 1u) ? 0x3715u : 0x6240u, sel_b = (qq & 2u) ? 0x3276u : 0x5410u;
#pragma unroll
        for (int cb = 0; cb < 4; ++cb) {
            const uint32_t mm = (cb < 2 ? p01 : p23) >> (16 * (cb & 1));
            const uint32_t cbyte = scale_byte(mm & 0xFFFFu);
            const uint64_t s2 = pack2(inv_scale_bits(cbyte), inv_scale_bits(cbyte));
            const uint32_t x = encode8(wc[cb][0], wc[cb][1], wc[cb][2], wc[cb][3], s2);
            const uint32_t a = __byte_perm(x, __shfl_xor_sync(0xFFFFFFFFu, x, 1), sel_a);
            const uint32_t y = __byte_perm(a, __shfl_xor_sync(0xFFFFFFFFu, a, 2), sel_b);
            const int64_t n = col + 8 * cb + (lane >> 2);
            sts32(qcol + (32 * c + 8 * cb + (lane >> 2)) * 16 + 4 * qq, y);
            if (qq == 0 && n < n_pad) {
                const int64_t atom = (n >> 7) * g.kb4o_col + (row0 >> 7);
                g.so_col[atom * 512 + (n & 31) * 16 + c * 4 + q] = static_cast<uint8_t>(n < g.N ? cbyte : 0u);
            }
        }
        return;
    }
    // The block that straddles M: column `lane` read down the staged rows, rows past M as 0.
    const int64_t n = col + lane;
    const uint32_t base = obuf + ((lane & 7u) << 1);
    uint32_t cw[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        uint32_t lo = lds_u16(base + swz64(2 * k, lane >> 3));
        uint32_t hi = lds_u16(base + swz64(2 * k + 1, lane >> 3));
        if (row0 + 2 * k >= g.M) lo = 0;
        if (row0 + 2 * k + 1 >= g.M) hi = 0;
        cw[k] = lo | (hi << 16);
    }
    uint32_t mc = cw[0];
#pragma unroll
    for (int i = 1; i < 16; ++i) mc = absmax2(mc, cw[i]);
    mc = absmax2(mc, mc >> 16) & 0x7FFFu;
    const uint32_t cbyte = scale_byte(mc);
    {
        const uint64_t s2 = pack2(inv_scale_bits(cbyte), inv_scale_bits(cbyte));
        sts128(qcol + (32 * c + lane) * 16, encode8(cw[0], cw[1], cw[2], cw[3], s2),
               encode8(cw[4], cw[5], cw[6], cw[7], s2), encode8(cw[8], cw[9], cw[10], cw[11], s2),
               encode8(cw[12], cw[13], cw[14], cw[15], s2));
    }
    if (n < n_pad) {
        const int64_t atom = (n >> 7) * g.kb4o_col + (row0 >> 7);
        g.so_col[atom * 512 + lane * 16 + c * 4 + q] = static_cast<uint8_t>(n < g.N ? cbyte : 0u);
    }
}

// Row tile mt2 and column tile nt of a problem's tile lt.  The tiles are walked in groups of
// g.group_m row tiles, the row tile fastest within a group: the clusters at work at one time
// share a few A row tiles and the group's B tiles, which L2 keeps.
__device__ __forceinline__ void pair_tile_coords(int lt, const GemmArgs& g, int* mt2, int* nt) {
    const int per_group = g.group_m * g.tiles_n;
    const int grp = lt / per_group;
    const int first = grp * g.group_m;
    const int gm = min(g.tiles_m2 - first, g.group_m);
    const int r = lt - grp * per_group;
    *mt2 = first + r % gm;
    *nt = r / gm;
}

// kBatched = false: one problem (P.count == 1); its arguments stay constant-bank operands,
// which the batched form's run-time problem index turns into registers (measured: the
// forward GEMM spilled and lost 4 us in the batched form).
// kBias: some problem of the launch carries a bias (the instance without one compiles the
// plain conversion only).
// kQuant: the epilogue also writes the MXFP4 blobs of C (one problem, bf16 through TMA).
// kWide: 256 x 384 tiles (PairCfg); every problem bf16 out through TMA stores, no kQuant.
template <bool kBatched, bool kBias, bool kQuant, bool kWide>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(PairCfg<kWide>::kThreads, 1)
    gemm_mxf4_pair_kernel(const __grid_constant__ GemmPairBatch P) {
    using C = PairCfg<kWide>;
    static_assert(!(kWide && kQuant), "output quantization runs on narrow tiles");
    constexpr int kStages = C::kStages;
    constexpr int kEpiWarps = C::kEpiWarps;
    extern __shared__ uint8_t smem_raw[];
    PairSmem<kWide>& sm = *reinterpret_cast<PairSmem<kWide>*>(
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
    // Problem of launch tile t, and t's index within that problem.
    auto task_of = [&](int t, int* local) {
        if (!kBatched) {
            *local = t;
            return 0;
        }
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
        mbar_init(smem_addr(&sm.tmem_full), 1);
        mbar_init(smem_addr(&sm.tmem_empty), 2 * kEpiWarps);
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
    cluster_sync_all();   // both CTAs' barriers exist before anything signals across
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
                prefetch_tensormap(&P.sfamap[j]);
                prefetch_tensormap(&P.sfbmap[j]);
            }
            const uint64_t pol = l2_policy_evict_last();
            int it = 0;
            bool ok = true;
            for (int t = cluster; t < num_tiles && ok; t += nclusters) {
                int lt;
                const int j = task_of(t, &lt);
                const GemmArgs& g = P.args[j];
                int mt2, nt;
                pair_tile_coords(lt, g, &mt2, &nt);
                const int arow = mt2 * 256 + static_cast<int>(rank) * 128;
                const int brow = nt * C::kTileN + static_cast<int>(rank) * 128;
                for (int ks = 0; ks < g.k_stages; ++ks, ++it) {
                    const int s = it % kStages;
                    const uint32_t ph = (it / kStages) & 1;
                    if (!mbar_wait(smem_addr(&sm.empty[s]), ph ^ 1, g.err, kErrGemmProducer, &sm.abort)) {
                        ok = false;
                        break;
                    }
                    if (leader) mbar_arrive_expect_tx(smem_addr(&sm.full[s]), 2 * C::kStageBytes);
                    const uint32_t bar = cluster_map(smem_addr(&sm.full[s]), 0);
                    tma_load_2d_pair(smem_addr(sm.a[s]), &P.amap[j], ks * BKB, arow, bar, pol);
                    tma_load_2d_pair(smem_addr(sm.b[s]), &P.bmap[j], ks * BKB, brow, bar, pol);
                    if (kWide)
                        tma_load_2d_pair(smem_addr(sm.b[s]) + 128 * BKB, &P.bmap2[j], ks * BKB,
                                         nt * C::kTileN + 256 + static_cast<int>(rank) * 64, bar, pol);
                    // Scale maps count 8-byte units: 2 atoms = 128 units per K step.
                    tma_load_2d_pair(smem_addr(sm.sfa[s]), &P.sfamap[j], ks * 128, 2 * mt2 + static_cast<int>(rank),
                                     bar, pol);
                    tma_load_2d_pair(smem_addr(sm.sfb[s]), &P.sfbmap[j], ks * 128, C::kBGroups * nt, bar, pol);
                }
            }
            // Drain (leader): every armed stage, both CTAs' bytes, has landed.
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
            int it = 0;
            bool ok = true;
            for (int t = cluster; t < num_tiles && ok; t += nclusters) {
                int lt;
                const GemmArgs& g = P.args[task_of(t, &lt)];
                for (int ks = 0; ks < g.k_stages; ++ks, ++it) {
                    if (!named_barrier_and(kBarHandoff, 64, true)) {
                        ok = false;
                        break;
                    }
                    if (elect_one()) {
                        tc_fence_after_sync();
                        const int s = it % kStages;
                        const int natoms = min(2, g.kb4 - 2 * ks);
                        // TMEM scale slot of the stage: A atoms a at columns 4a, then per atom a
                        // the B groups gb at 8 + 4 (kBGroups a + gb)
                        const uint32_t sf = tmem + C::kSfTmemBase + s * C::kSfTmemPerStage;
                        const uint32_t sfa_s = smem_addr(sm.sfa[s]);
                        const uint32_t sfb_s = smem_addr(sm.sfb[s]);
                        const uint64_t adesc = smem_desc(smem_addr(sm.a[s]), 16, 1024, 2);
                        const uint64_t bdesc = smem_desc(smem_addr(sm.b[s]), 16, 1024, 2);
                        const uint64_t bdesc2 = smem_desc(smem_addr(sm.b[s]) + 128 * BKB, 16, 1024, 2);
                        // per scale atom (128 elements of K): its copies, then the two K-64
                        // slices that read them, so a tile's first MMA waits for one atom's
                        // copies only
                        for (int a = 0; a < natoms; ++a) {
                            tc_cp_32x128b_warpx4_pair(sf + a * 4, smem_desc(sfa_s + a * 512, 0, 128, 0));
#pragma unroll
                            for (int gb = 0; gb < C::kBGroups; ++gb)
                                tc_cp_32x128b_warpx4_pair(sf + 8 + (a * C::kBGroups + gb) * 4,
                                                          smem_desc(sfb_s + gb * 1024 + a * 512, 0, 128, 0));
                            const uint32_t sfb = sf + 8 + a * 4 * C::kBGroups;
#pragma unroll
                            for (int jj = 0; jj < 2; ++jj) {
                                const int j = 2 * a + jj;
                                const uint32_t sf_id = jj * 2;
                                tc_mma_mxf4_pair(tmem, adesc + 2 * j, bdesc + 2 * j, pair_idesc(sf_id, 256), sf + a * 4,
                                                 sfb, (ks | j) != 0);
                                if (kWide)
                                    tc_mma_mxf4_pair(tmem + 256, adesc + 2 * j, bdesc2 + 2 * j, pair_idesc(sf_id, 128),
                                                     sf + a * 4, sfb + 8, (ks | j) != 0);
                            }
                        }
                        tc_commit_pair_multicast(smem_addr(&sm.empty[s]), 3);
                        if (ks == g.k_stages - 1) tc_commit_pair_multicast(smem_addr(&sm.tmem_full), 3);
                    }
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
                const GemmArgs& g = P.args[task_of(t, &lt)];
                for (int ks = 0; ks < g.k_stages; ++ks, ++it) {
                    int w = 1;
                    if (lane == 0) {
                        if (ks == 0 && tl > 0)
                            w = mbar_wait(smem_addr(&sm.tmem_empty), (tl - 1) & 1, g.err, kErrGemmMma, &sm.abort);
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
        const uint32_t qrow_buf = kQuant ? smem_addr(sm.qrow[warp - kEpi0]) : 0u;
        const uint32_t qcol_buf = kQuant ? smem_addr(sm.qcol[warp - kEpi0]) : 0u;
        const uint64_t pol = l2_policy_evict_first();
        const uint32_t leader_tmem_empty = cluster_map(smem_addr(&sm.tmem_empty), 0);
        if (lane == 0) {
            for (int j = 0; j < P.count; ++j)
                if (P.args[j].c_tma) prefetch_tensormap(&P.cmap[j]);
            if (kQuant) {
                prefetch_tensormap(&P.qrowmap);
                if (P.args[0].qo_col != nullptr) prefetch_tensormap(&P.qcolmap);
            }
        }
        int tl = 0;
        for (int t = cluster; t < num_tiles; t += nclusters, ++tl) {
            int okw = 1;
            if (warp == kEpi0 && lane == 0)
                okw = mbar_wait(smem_addr(&sm.tmem_full), tl & 1, err, kErrGemmEpilogue, &sm.abort);
            if (!named_barrier_and(kBarEpilogue, kEpiWarps * 32, __shfl_sync(0xFFFFFFFFu, okw, 0) != 0)) break;
            tc_fence_after_sync();
            const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + h * 128;
            if (kWide) {
                // bf16 through TMA stores.  The accumulator is read in two halves of 64
                // columns, the first converted to bf16 pairs while the second is read, so no
                // more than 64 fp32 values are live (the 480-thread CTA has 128 registers a
                // thread); the accumulator is released as soon as the second half is in.
                int lt;
                const int pj = task_of(t, &lt);
                const GemmArgs& g = P.args[pj];
                int mt2, nt;
                pair_tile_coords(lt, g, &mt2, &nt);
                const int64_t rowblk = static_cast<int64_t>(mt2) * 256 + rank * 128;
                const int64_t col0 = static_cast<int64_t>(nt) * C::kTileN + h * 128;
                const uint16_t* const bias = kBias ? g.bias : nullptr;
                uint32_t wb[4][16];
                {
                    uint32_t v0[32], v1[32];
                    tc_ld_32x32b_x32(taddr + 0, v0);
                    tc_ld_32x32b_x32(taddr + 32, v1);
                    tc_wait_ld();
                    convert_piece<false>(v0, bias, col0, g.N, wb[0]);
                    convert_piece<false>(v1, bias, col0 + 32, g.N, wb[1]);
                    // the first half's bf16 pairs exist before the second half is read
#pragma unroll
                    for (int i = 0; i < 16; ++i) asm volatile("" : "+r"(wb[0][i]), "+r"(wb[1][i]));
                    tc_ld_32x32b_x32(taddr + 64, v0);
                    tc_ld_32x32b_x32(taddr + 96, v1);
                    tc_wait_ld();
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster_relaxed(leader_tmem_empty);
                    convert_piece<false>(v0, bias, col0 + 64, g.N, wb[2]);
                    convert_piece<false>(v1, bias, col0 + 96, g.N, wb[3]);
                }
                // The four warps of column group h (one per lane quarter) stage their 32 x 32
                // pieces side by side, in row order, and one of them stores the 128-row column
                // strip with one tensor store (a quarter of the store operations).
                if (rowblk >= g.M || col0 >= g.N) continue;   // the same for the group's warps
                const uint32_t gbuf = smem_addr(sm.out[4 * h]);
                const bool issuer = ((warp - kEpi0) & 3) == 0;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    if (col0 + c * 32 >= g.N) break;
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        sts128(gbuf + q * kOutBytes + swz64(lane, j), wb[c][4 * j], wb[c][4 * j + 1], wb[c][4 * j + 2],
                               wb[c][4 * j + 3]);
                    fence_proxy_async_smem();
                    named_barrier(kBarStore0 + h, 128);
                    if (issuer && lane == 0) {
                        tma_store_2d_hint(&P.cmap[pj], static_cast<int32_t>(col0 + c * 32), static_cast<int32_t>(rowblk),
                                          gbuf, pol);
                        bulk_commit_group();
                        bulk_wait_read_all();
                    }
                    named_barrier(kBarStore0 + h, 128);
                }
                continue;
            }
            uint32_t v[4][32];
            tc_ld_32x32b_x32(taddr + 0, v[0]);
            tc_ld_32x32b_x32(taddr + 32, v[1]);
            tc_ld_32x32b_x32(taddr + 64, v[2]);
            tc_ld_32x32b_x32(taddr + 96, v[3]);
            tc_wait_ld();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster_relaxed(leader_tmem_empty);

            int lt;
            const int pj = task_of(t, &lt);
            const GemmArgs& g = P.args[pj];
            int mt2, nt;
            pair_tile_coords(lt, g, &mt2, &nt);
            const int64_t row0 = static_cast<int64_t>(mt2) * 256 + rank * 128 + q * 32;
            const int64_t col0 = static_cast<int64_t>(nt) * 256 + h * 128;
            if (kQuant) {
                // Output quantization (bf16 through TMA stores): the warps of padding rows, up
                // to M's 128-row padding, still write their zero scale bytes.  The four pieces
                // are converted to bf16 first, which frees the fp32 accumulator registers.
                if (row0 >= ((g.M + 127) & ~int64_t{127}) || col0 >= g.N) continue;
                uint32_t wb[4][16];
                const uint16_t* const bias = kBias ? g.bias : nullptr;
#pragma unroll
                for (int c = 0; c < 4; ++c) convert_piece<false>(v[c], bias, col0 + c * 32, g.N, wb[c]);
                uint32_t srow = 0;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    if (lane == 0) bulk_wait_read_all();
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        sts128(obuf + swz64(lane, j), wb[c][4 * j], wb[c][4 * j + 1], wb[c][4 * j + 2], wb[c][4 * j + 3]);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0 && row0 < g.M && col0 + c * 32 < g.N) {
                        tma_store_2d_hint(&P.cmap[pj], static_cast<int32_t>(col0 + c * 32), static_cast<int32_t>(row0),
                                          obuf, pol);
                        bulk_commit_group();
                    }
                    quantize_out_piece(g, wb[c], obuf, qrow_buf, qcol_buf, row0, col0 + c * 32, c, q, lane, &srow);
                }
                // the row's 4 scale bytes of this 128-column half, one word
                const int64_t atom = ((row0 + lane) >> 7) * g.kb4o_row + (col0 >> 7);
                *reinterpret_cast<uint32_t*>(g.so_row + atom * 512 + lane * 16 + q * 4) = srow;
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    if (row0 < g.M)
                        tma_store_2d_hint(&P.qrowmap, static_cast<int32_t>(col0 >> 1), static_cast<int32_t>(row0),
                                          qrow_buf, pol);
                    if (g.qo_col != nullptr)
                        tma_store_2d_hint(&P.qcolmap, static_cast<int32_t>(row0 >> 1), static_cast<int32_t>(col0),
                                          qcol_buf, pol);
                    bulk_commit_group();
                }
                continue;
            }
            if (row0 >= g.M || col0 >= g.N) continue;
            if (g.c_tma) {
                const int per = g.out_f32 ? 16 : 32;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    if (c * per >= 128 || col0 + c * per >= g.N) break;
                    if (lane == 0) bulk_wait_read_all();
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
        if (lane == 0) bulk_wait_all();
        __syncwarp();
    }

    tc_fence_before_sync();
    __syncthreads();
    cluster_sync_all();   // no CTA leaves or frees TMEM while its peer may still use it
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc_pair(tmem, kTmemCols);
    }
}

}  // namespace

size_t gemm_pair_smem_bytes(bool wide) {
    return (wide ? sizeof(PairSmem<true>) : sizeof(PairSmem<false>)) + 1024;
}

int gemm_pair_max_clusters(bool wide) {
    static int cached[2][64] = {{0}};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cached[wide][dev] > 0) return cached[wide][dev];
    const size_t smem = gemm_pair_smem_bytes(wide);
    auto kernel = wide ? gemm_mxf4_pair_kernel<true, true, false, true> : gemm_mxf4_pair_kernel<true, true, false, false>;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(wide ? PairCfg<true>::kThreads : PairCfg<false>::kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) return 0;
    cached[wide][dev] = n;
    return n;
}

cudaError_t launch_gemm_pair(const GemmPairBatch& b, int clusters, cudaStream_t stream, bool quant, bool wide) {
    const size_t smem = gemm_pair_smem_bytes(wide);
    bool bias = false;
    for (int j = 0; j < b.count; ++j) bias = bias || b.args[j].bias != nullptr;
    if (quant && (wide || b.count != 1 || b.args[0].out_f32 || !b.args[0].c_tma || b.args[0].qo_row == nullptr))
        return cudaErrorInvalidValue;
    if (wide)
        for (int j = 0; j < b.count; ++j)
            if (b.args[j].out_f32 || !b.args[j].c_tma) return cudaErrorInvalidValue;
    using K = void (*)(GemmPairBatch);
    K kernel;
    if (quant)
        kernel = bias ? gemm_mxf4_pair_kernel<false, true, true, false> : gemm_mxf4_pair_kernel<false, false, true, false>;
    else if (wide)
        kernel = b.count > 1 ? (bias ? gemm_mxf4_pair_kernel<true, true, false, true> : gemm_mxf4_pair_kernel<true, false, false, true>)
                             : (bias ? gemm_mxf4_pair_kernel<false, true, false, true> : gemm_mxf4_pair_kernel<false, false, false, true>);
    else
        kernel = b.count > 1 ? (bias ? gemm_mxf4_pair_kernel<true, true, false, false> : gemm_mxf4_pair_kernel<true, false, false, false>)
                             : (bias ? gemm_mxf4_pair_kernel<false, true, false, false> : gemm_mxf4_pair_kernel<false, false, false, false>);
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * clusters, 1, 1);
    cfg.blockDim = dim3(wide ? PairCfg<true>::kThreads : PairCfg<false>::kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, b);
}

}  // namespace mxfp4
