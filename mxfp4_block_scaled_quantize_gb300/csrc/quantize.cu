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
// thread streams tiles into a 3-stage shared-memory ring with TMA (out-of-bounds rows and
// columns arrive as zeros, which is exactly the padding rule); 8 consumer warps quantize
// each tile twice from shared memory -- rowwise with 16-byte vector reads and a 4-lane
// shuffle amax, columnwise with each thread owning a column pair of one 32-row block --
// so X is read from HBM once for both packings.  The scale bytes of a tile form exactly
// one 512-byte atom of the tensor-core scale layout per packing; they are gathered in
// shared memory and written with 16-byte stores.
#include <cuda_bf16.h>

#include "launch.h"
#include "ptx.cuh"

namespace mxfp4 {
namespace {

constexpr int kQT = 128;                       // tile edge (rows and columns)
constexpr int kQStages = 3;
constexpr int kQConsumerWarps = 8;
constexpr int kQConsumers = kQConsumerWarps * 32;
constexpr int kQThreads = kQConsumers + 32;    // + one producer warp
constexpr int kQTileBytes = kQT * kQT * 2;
constexpr int kQRowPitch = kQT * 2;            // bytes per tile row in shared memory
constexpr int kQCtasPerSm = 2;

struct QuantSmem {
    uint8_t tile[kQStages][kQTileBytes];
    uint8_t atom_row[2][512];
    uint8_t atom_col[2][512];
    uint64_t full[kQStages];
    uint64_t empty[kQStages];
    int abort;
    int ok;
};

__device__ __forceinline__ float lo_f(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_f(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// E8M0 byte of a block from the bit pattern of its largest magnitude (sign cleared).
__device__ __forceinline__ uint32_t scale_byte(uint32_t amax_bits) {
    const int ef = static_cast<int>(amax_bits >> 7);
    return static_cast<uint32_t>(ef > 2 ? ef - 2 : 0);
}

// 2^(127 - byte) as fp32: always a normal number for byte in [0, 252].
__device__ __forceinline__ float inv_scale(uint32_t byte) { return __uint_as_float((254u - byte) << 23); }

// Two fp32 values -> one byte of two E2M1 codes, `lo` in the low nibble.
__device__ __forceinline__ uint32_t cvt_e2m1x2(float hi, float lo) {
    uint32_t r;
    asm("{\n\t.reg .b8 t;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
        "cvt.u32.u8 %0, t;\n\t}"
        : "=r"(r)
        : "f"(hi), "f"(lo));
    return r;
}

// Sign bits of the two bf16 in w placed at bits 3 and 7 (the sign bits of the byte's two
// nibbles): negative inputs that round to zero keep their sign as 0x8.
__device__ __forceinline__ uint32_t sign_pair_lo_hi(uint32_t w) {
    return ((w >> 12) & 0x8u) | ((w >> 24) & 0x80u);
}

template <bool kSignFix>
__device__ __forceinline__ uint32_t encode8(const uint4& w, float s) {
    uint32_t b0 = cvt_e2m1x2(hi_f(w.x) * s, lo_f(w.x) * s);
    uint32_t b1 = cvt_e2m1x2(hi_f(w.y) * s, lo_f(w.y) * s);
    uint32_t b2 = cvt_e2m1x2(hi_f(w.z) * s, lo_f(w.z) * s);
    uint32_t b3 = cvt_e2m1x2(hi_f(w.w) * s, lo_f(w.w) * s);
    uint32_t q = b0 | (b1 << 8) | (b2 << 16) | (b3 << 24);
    if (kSignFix) {
        q |= sign_pair_lo_hi(w.x) | (sign_pair_lo_hi(w.y) << 8) | (sign_pair_lo_hi(w.z) << 16) |
             (sign_pair_lo_hi(w.w) << 24);
    }
    return q;
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

template <bool kDual, bool kSignFix>
__global__ void __launch_bounds__(kQThreads, kQCtasPerSm)
    quantize_kernel(const __grid_constant__ CUtensorMap xmap, const QuantArgs p) {
    extern __shared__ uint8_t smem_raw[];
    QuantSmem& sm = *reinterpret_cast<QuantSmem*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~static_cast<uintptr_t>(127));

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int num_tiles = p.tiles_m * p.tiles_k;

    if (tid == 0) {
        for (int s = 0; s < kQStages; ++s) {
            mbar_init(smem_addr(&sm.full[s]), 1);
            mbar_init(smem_addr(&sm.empty[s]), 1);
        }
        sm.abort = 0;
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == kQConsumerWarps) {
        // ------------------------------------------------------------- producer (TMA)
        if (lane_id() == 0) {
            prefetch_tensormap(&xmap);
            int it = 0;
            for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++it) {
                const int s = it % kQStages;
                const uint32_t ph = (it / kQStages) & 1;
                if (!mbar_wait(smem_addr(&sm.empty[s]), ph ^ 1, p.err, kErrQuantProducer, &sm.abort))
                    break;
                const int tm = t / p.tiles_k, tk = t % p.tiles_k;
                mbar_arrive_expect_tx(smem_addr(&sm.full[s]), kQTileBytes);
                tma_load_2d(smem_addr(sm.tile[s]), &xmap, tk * kQT, tm * kQT, smem_addr(&sm.full[s]));
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
    int it = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++it) {
        const int s = it % kQStages;
        const uint32_t ph = (it / kQStages) & 1;
        const int buf = it & 1;
        if (tid == 0)
            sm.ok = mbar_wait(smem_addr(&sm.full[s]), ph, p.err, kErrQuantConsumer, &sm.abort) ? 1 : 0;
        named_barrier(1, kQConsumers);
        if (!*reinterpret_cast<volatile int*>(&sm.ok)) break;

        const int tm = t / p.tiles_k, tk = t % p.tiles_k;
        const int64_t m0 = static_cast<int64_t>(tm) * kQT;
        const int64_t k0 = static_cast<int64_t>(tk) * kQT;
        const uint32_t tile = smem_addr(sm.tile[s]);

        // ---- rowwise: 2048 chunks of 8 bf16; 4 consecutive chunks form one block
#pragma unroll 2
        for (int i = 0; i < (kQT * kQT / 8) / kQConsumers; ++i) {
            const int id = i * kQConsumers + tid;
            const int r = id >> 4, c = id & 15;
            const uint4 w = lds128(tile + r * kQRowPitch + c * 16);
            uint32_t m = __vmaxu2(__vmaxu2(w.x & 0x7FFF7FFFu, w.y & 0x7FFF7FFFu),
                                  __vmaxu2(w.z & 0x7FFF7FFFu, w.w & 0x7FFF7FFFu));
            m = max(m & 0xFFFFu, m >> 16);
            m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
            m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
            const uint32_t byte = scale_byte(m);
            const uint32_t q = encode8<kSignFix>(w, inv_scale(byte));
            const int64_t row = m0 + r;
            if (row < p.M)
                *reinterpret_cast<uint32_t*>(p.q_row + row * p.ldq_row + (k0 >> 1) + c * 4) = q;
            if ((c & 3) == 0) {
                const int cb = c >> 2;
                const int pos = p.tc_layout ? ((r & 31) * 16 + (r >> 5) * 4 + cb) : (r * 4 + cb);
                sm.atom_row[buf][pos] = static_cast<uint8_t>(byte);
            }
        }

        // ---- columnwise: thread owns columns (2pc, 2pc+1) of the 32-row block rb
        if (kDual) {
            const int pc = tid & 63, rb = tid >> 6;
            uint32_t w[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) w[i] = lds32(tile + (rb * 32 + i) * kQRowPitch + pc * 4);
            uint32_t m = 0;
#pragma unroll
            for (int i = 0; i < 32; ++i) m = __vmaxu2(m, w[i] & 0x7FFF7FFFu);
            const uint32_t byte0 = scale_byte(m & 0xFFFFu), byte1 = scale_byte(m >> 16);
            const float s0 = inv_scale(byte0), s1 = inv_scale(byte1);
            uint32_t q0[4] = {0, 0, 0, 0}, q1[4] = {0, 0, 0, 0};
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const uint32_t a = w[2 * j], b = w[2 * j + 1];
                uint32_t c0 = cvt_e2m1x2(lo_f(b) * s0, lo_f(a) * s0);
                uint32_t c1 = cvt_e2m1x2(hi_f(b) * s1, hi_f(a) * s1);
                if (kSignFix) {
                    c0 |= ((a >> 12) & 0x8u) | ((b >> 8) & 0x80u);
                    c1 |= ((a >> 28) & 0x8u) | ((b >> 24) & 0x80u);
                }
                q0[j >> 2] |= c0 << (8 * (j & 3));
                q1[j >> 2] |= c1 << (8 * (j & 3));
            }
            const int64_t kc = k0 + 2 * pc;
            const int64_t off = (m0 + rb * 32) >> 1;
            if (kc < p.K)
                *reinterpret_cast<uint4*>(p.q_col + kc * p.ldq_col + off) =
                    make_uint4(q0[0], q0[1], q0[2], q0[3]);
            if (kc + 1 < p.K)
                *reinterpret_cast<uint4*>(p.q_col + (kc + 1) * p.ldq_col + off) =
                    make_uint4(q1[0], q1[1], q1[2], q1[3]);
            const int kl0 = 2 * pc, kl1 = 2 * pc + 1;
            if (p.tc_layout) {
                sm.atom_col[buf][(kl0 & 31) * 16 + (kl0 >> 5) * 4 + rb] = static_cast<uint8_t>(byte0);
                sm.atom_col[buf][(kl1 & 31) * 16 + (kl1 >> 5) * 4 + rb] = static_cast<uint8_t>(byte1);
            } else {
                sm.atom_col[buf][kl0 * 4 + rb] = static_cast<uint8_t>(byte0);
                sm.atom_col[buf][kl1 * 4 + rb] = static_cast<uint8_t>(byte1);
            }
        }

        // All reads of the stage and all scale bytes of the tile are done.
        named_barrier(1, kQConsumers);
        if (tid == 0) mbar_arrive(smem_addr(&sm.empty[s]));

        if (p.tc_layout) {
            if (tid < 32) {
                const int64_t atom = static_cast<int64_t>(tm) * (p.kb_row >> 2) + tk;
                *reinterpret_cast<uint4*>(p.s_row + atom * 512 + tid * 16) =
                    *reinterpret_cast<const uint4*>(&sm.atom_row[buf][tid * 16]);
            } else if (kDual && tid < 64) {
                const int64_t atom = static_cast<int64_t>(tk) * (p.kb_col >> 2) + tm;
                *reinterpret_cast<uint4*>(p.s_col + atom * 512 + (tid - 32) * 16) =
                    *reinterpret_cast<const uint4*>(&sm.atom_col[buf][(tid - 32) * 16]);
            }
        } else {
            if (tid < kQT) {
                const int64_t row = m0 + tid;
                if (row < p.M)
                    *reinterpret_cast<uint32_t*>(p.s_row + row * p.kb_row + (k0 >> 5)) =
                        *reinterpret_cast<const uint32_t*>(&sm.atom_row[buf][tid * 4]);
            } else if (kDual) {
                const int64_t kr = k0 + (tid - kQT);
                if (kr < p.K)
                    *reinterpret_cast<uint32_t*>(p.s_col + kr * p.kb_col + (m0 >> 5)) =
                        *reinterpret_cast<const uint32_t*>(&sm.atom_col[buf][(tid - kQT) * 4]);
            }
        }
    }
}

// Negative values that round to zero must come out as -0 (0x8).  Whether the hardware
// conversion keeps that sign is checked by the parity tests; the explicit sign merge is
// exact either way and is kept on.
constexpr bool kSignFixDefault = true;

}  // namespace

size_t quantize_smem_bytes() { return sizeof(QuantSmem) + 128; }
int quantize_ctas_per_sm() { return kQCtasPerSm; }

cudaError_t launch_quantize(const CUtensorMap& xmap, const QuantArgs& a, bool dual, int grid,
                            cudaStream_t stream) {
    const size_t smem = quantize_smem_bytes();
    if (dual) {
        auto k = quantize_kernel<true, kSignFixDefault>;
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        k<<<grid, kQThreads, smem, stream>>>(xmap, a);
    } else {
        auto k = quantize_kernel<false, kSignFixDefault>;
        cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        k<<<grid, kQThreads, smem, stream>>>(xmap, a);
    }
    return cudaGetLastError();
}

}  // namespace mxfp4
