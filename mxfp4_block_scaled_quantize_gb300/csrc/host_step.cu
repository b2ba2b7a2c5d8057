// host_step.cu -- mxfp4_linear_step_host: one step of MXFP4 linears from host buffers to
// host buffers (include/mxfp4.h).  Host code only: it carves the caller's workspace, copies
// the inputs in on one library-owned stream, launches the library's quantizer and GEMM
// entry points on the caller's stream, and copies every result out on a second stream as
// soon as the kernel that writes it is done.  Events order the three streams, so each
// quantization waits only for its own inputs and the result copies overlap later kernels.
// The pipelined form (mxfp4_linear_step_host_pipelined) also lets consecutive steps
// overlap: a step's results leave from one of two output sets while the next step's inputs
// come in and its kernels run.
#include <cuda_runtime.h>

#include <cstring>
#include <mutex>

#include "mxfp4.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kEventsPerStep = 4 * MXFP4_MAX_BATCH + 3;
constexpr int64_t kMaxDim = (int64_t{1} << 31) - 512;

struct CopyStreams {
    bool ready = false;
    cudaStream_t h2d = nullptr;
    cudaStream_t d2h = nullptr;
    cudaEvent_t ev[kEventsPerStep] = {};
    // Across calls: the last step's quantizers are done with each linear's device inputs
    // (X and W; dY), so the next step may refill them; and the copies out of the last step
    // that wrote each output set are done, so a step may write that set again.
    cudaEvent_t consumed_xw[MXFP4_MAX_BATCH] = {};
    cudaEvent_t consumed_dy[MXFP4_MAX_BATCH] = {};
    cudaEvent_t slot_free[2] = {};
    bool consumed_valid = false;
    bool slot_valid[2] = {false, false};
    int slot = 0;
};

std::mutex g_host_mutex;
CopyStreams g_copy[kMaxDevices];

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int64_t pad128(int64_t n) { return cdiv(n, 128) * 128; }
inline int64_t round8(int64_t n) { return cdiv(n, 8) * 8; }
inline size_t align256(size_t n) { return (n + 255) & ~static_cast<size_t>(255); }

// Device buffers of one linear, carved from the workspace in this order.
struct Carve {
    uint8_t* xd;  // bf16 X, row pitch round8(K)
    uint8_t* wd;  // bf16 W, row pitch round8(K)
    uint8_t* dyd; // bf16 dY, row pitch round8(N)
    uint8_t *xrq, *xrs, *wrq, *wrs;                  // row blobs of X and W
    uint8_t *xcq, *xcs, *wcq, *wcs, *drq, *drs, *dcq, *dcs;   // col blobs, dY's blobs
    uint8_t *y, *dx, *dw;
};

size_t blob_q(int64_t rows, int64_t k) { return static_cast<size_t>(rows) * static_cast<size_t>(pad128(k) / 2); }
size_t blob_s(int64_t rows, int64_t k) { return static_cast<size_t>(pad128(rows)) * static_cast<size_t>(pad128(k) / 32); }

// Lays out one task's output buffers (Y; dX, dW) from `base` (nullptr: only measures) over
// the ones `carve` placed.  Returns the bytes used.
size_t carve_outputs(const mxfp4_linear_host_task& t, uint8_t* base, Carve* c) {
    size_t off = 0;
    auto take = [&](size_t n) {
        uint8_t* p = base ? base + off : nullptr;
        off += align256(n);
        return p;
    };
    const size_t es = t.out_dtype == MXFP4_OUT_F32 ? 4 : 2;
    c->y = take(static_cast<size_t>(t.M) * t.N * es);
    if (t.train) {
        c->dx = take(static_cast<size_t>(t.M) * t.K * es);
        c->dw = take(static_cast<size_t>(t.N) * t.K * es);
    }
    return off;
}

// Lays out one task's buffers from `base` (nullptr: only measures).  Returns the bytes used.
size_t carve(const mxfp4_linear_host_task& t, uint8_t* base, Carve* c) {
    size_t off = 0;
    auto take = [&](size_t n) {
        uint8_t* p = base ? base + off : nullptr;
        off += align256(n);
        return p;
    };
    const size_t es = t.out_dtype == MXFP4_OUT_F32 ? 4 : 2;
    const int64_t M = t.M, N = t.N, K = t.K;
    c->xd = take(static_cast<size_t>(M) * round8(K) * 2);
    c->wd = take(static_cast<size_t>(N) * round8(K) * 2);
    c->xrq = take(blob_q(M, K));
    c->xrs = take(blob_s(M, K));
    c->wrq = take(blob_q(N, K));
    c->wrs = take(blob_s(N, K));
    c->y = take(static_cast<size_t>(M) * N * es);
    if (t.train) {
        c->dyd = take(static_cast<size_t>(M) * round8(N) * 2);
        c->xcq = take(blob_q(K, M));
        c->xcs = take(blob_s(K, M));
        c->wcq = take(blob_q(K, N));
        c->wcs = take(blob_s(K, N));
        c->drq = take(blob_q(M, N));
        c->drs = take(blob_s(M, N));
        c->dcq = take(blob_q(N, M));
        c->dcs = take(blob_s(N, M));
        c->dx = take(static_cast<size_t>(M) * K * es);
        c->dw = take(static_cast<size_t>(N) * K * es);
    }
    return off;
}

// Shapes, dtype and mode of every task; with `pointers`, also the host buffers.
mxfp4_status check_tasks(int32_t count, const mxfp4_linear_host_task* tasks, bool pointers) {
    if (count < 1 || count > MXFP4_MAX_BATCH || tasks == nullptr) return MXFP4_ERR_INVALID_ARG;
    for (int i = 0; i < count; ++i) {
        const mxfp4_linear_host_task& t = tasks[i];
        if (t.M < 1 || t.N < 1 || t.K < 1 || t.M > kMaxDim || t.N > kMaxDim || t.K > kMaxDim)
            return MXFP4_ERR_INVALID_ARG;
        if (t.out_dtype != MXFP4_OUT_BF16 && t.out_dtype != MXFP4_OUT_F32) return MXFP4_ERR_INVALID_ARG;
        if (t.train != 0 && t.train != 1) return MXFP4_ERR_INVALID_ARG;
        if (pointers && (!t.x || !t.w || !t.y)) return MXFP4_ERR_INVALID_ARG;
        if (pointers && t.train && (!t.dy || !t.dx || !t.dw)) return MXFP4_ERR_INVALID_ARG;
    }
    return MXFP4_OK;
}

size_t total_bytes(int32_t count, const mxfp4_linear_host_task* tasks) {
    size_t n = 0;
    Carve c = {};
    for (int i = 0; i < count; ++i) n += carve(tasks[i], nullptr, &c);
    return n;
}

// The pipelined step's workspace: the plain step's, then a second set of outputs.
size_t pipelined_bytes(int32_t count, const mxfp4_linear_host_task* tasks) {
    size_t n = total_bytes(count, tasks);
    Carve c = {};
    for (int i = 0; i < count; ++i) n += carve_outputs(tasks[i], nullptr, &c);
    return n;
}

// bf16 rows of `cols` elements from dense host rows into device rows of pitch round8(cols).
cudaError_t copy_in(uint8_t* dst, const void* src, int64_t rows, int64_t cols, cudaStream_t s) {
    const size_t w = static_cast<size_t>(cols) * 2;
    const size_t dp = static_cast<size_t>(round8(cols)) * 2;
    if (dp == w) return cudaMemcpyAsync(dst, src, w * rows, cudaMemcpyHostToDevice, s);
    return cudaMemcpy2DAsync(dst, dp, src, w, w, static_cast<size_t>(rows), cudaMemcpyHostToDevice, s);
}

cudaError_t copy_out(void* dst, const uint8_t* src, int64_t rows, int64_t cols, size_t es, cudaStream_t s) {
    return cudaMemcpyAsync(dst, src, static_cast<size_t>(rows) * cols * es, cudaMemcpyDeviceToHost, s);
}

mxfp4_status copy_streams(CopyStreams** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MXFP4_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return MXFP4_ERR_UNSUPPORTED_DEVICE;
    CopyStreams& c = g_copy[dev];
    if (!c.ready) {
        if (cudaStreamCreateWithFlags(&c.h2d, cudaStreamNonBlocking) != cudaSuccess ||
            cudaStreamCreateWithFlags(&c.d2h, cudaStreamNonBlocking) != cudaSuccess)
            return MXFP4_ERR_CUDA;
        for (auto& e : c.ev)
            if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return MXFP4_ERR_CUDA;
        for (int i = 0; i < MXFP4_MAX_BATCH; ++i)
            if (cudaEventCreateWithFlags(&c.consumed_xw[i], cudaEventDisableTiming) != cudaSuccess ||
                cudaEventCreateWithFlags(&c.consumed_dy[i], cudaEventDisableTiming) != cudaSuccess)
                return MXFP4_ERR_CUDA;
        for (auto& e : c.slot_free)
            if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return MXFP4_ERR_CUDA;
        c.ready = true;
    }
    *out = &c;
    return MXFP4_OK;
}

#define MX_TRY(x)                                      \
    do {                                               \
        if ((x) != cudaSuccess) return MXFP4_ERR_CUDA; \
    } while (0)
#define MX_TRY_ST(x)                        \
    do {                                    \
        const mxfp4_status st_ = (x);       \
        if (st_ != MXFP4_OK) return st_;    \
    } while (0)

}  // namespace

namespace {

// One step from host buffers to host buffers (both entry points).  Pipelined: the
// workspace holds two output sets used alternately, each refill of a device input waits
// only for the previous step's quantizer of that input, and the caller's stream is not
// ordered after the copies out (mxfp4_linear_host_wait does that).
mxfp4_status step_host(int32_t count, const mxfp4_linear_host_task* tasks, void* workspace, size_t workspace_bytes,
                       mxfp4_stream_t stream, bool pipelined) {
    MX_TRY_ST(check_tasks(count, tasks, true));
    if (workspace == nullptr ||
        workspace_bytes < (pipelined ? pipelined_bytes(count, tasks) : total_bytes(count, tasks)))
        return MXFP4_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MXFP4_ERR_MISALIGNED;
    std::lock_guard<std::mutex> lock(g_host_mutex);
    CopyStreams* cs = nullptr;
    MX_TRY_ST(copy_streams(&cs));
    cudaStream_t comp = reinterpret_cast<cudaStream_t>(stream);
    cudaEvent_t* ev = cs->ev;
    // ev[0]: step start; ev[1 + 4i ..]: X/W in, dY in, Y ready, dX/dW ready; last two: copies done.
    cudaEvent_t& ev_start = ev[0];
    auto ev_xw = [&](int i) -> cudaEvent_t& { return ev[1 + 4 * i]; };
    auto ev_dy = [&](int i) -> cudaEvent_t& { return ev[2 + 4 * i]; };
    auto ev_y = [&](int i) -> cudaEvent_t& { return ev[3 + 4 * i]; };
    auto ev_bwd = [&](int i) -> cudaEvent_t& { return ev[4 + 4 * i]; };
    cudaEvent_t& ev_h2d_done = ev[kEventsPerStep - 2];
    cudaEvent_t& ev_d2h_done = ev[kEventsPerStep - 1];

    Carve c[MXFP4_MAX_BATCH] = {};
    uint8_t* base = static_cast<uint8_t*>(workspace);
    for (int i = 0; i < count; ++i) base += carve(tasks[i], base, &c[i]);
    const int slot = pipelined ? cs->slot : 0;
    if (slot == 1)   // the second output set, after the first layout
        for (int i = 0; i < count; ++i) base += carve_outputs(tasks[i], base, &c[i]);
    const bool wait_inputs = pipelined && cs->consumed_valid;

    // The previous step's kernels are done with the input buffers before they refill
    // (pipelined: each input waits only for the quantizer that read it).
    MX_TRY(cudaEventRecord(ev_start, comp));
    if (!pipelined) MX_TRY(cudaStreamWaitEvent(cs->h2d, ev_start, 0));
    MX_TRY(cudaStreamWaitEvent(cs->d2h, ev_start, 0));
    // The output set is free: the copies out of the step that last wrote it are done (a
    // plain step after pipelined ones waits for all their copies out).
    if (pipelined && cs->slot_valid[slot]) MX_TRY(cudaStreamWaitEvent(comp, cs->slot_free[slot], 0));
    if (!pipelined && (cs->slot_valid[0] || cs->slot_valid[1])) MX_TRY(cudaStreamWaitEvent(comp, ev_d2h_done, 0));
    // Inputs in the order the kernels read them: X, W of each forward, then dY of each
    // backward (reverse task order).
    for (int i = 0; i < count; ++i) {
        const mxfp4_linear_host_task& t = tasks[i];
        if (wait_inputs) MX_TRY(cudaStreamWaitEvent(cs->h2d, cs->consumed_xw[i], 0));
        MX_TRY(copy_in(c[i].xd, t.x, t.M, t.K, cs->h2d));
        MX_TRY(copy_in(c[i].wd, t.w, t.N, t.K, cs->h2d));
        MX_TRY(cudaEventRecord(ev_xw(i), cs->h2d));
    }
    for (int i = count - 1; i >= 0; --i) {
        const mxfp4_linear_host_task& t = tasks[i];
        if (!t.train) continue;
        if (wait_inputs) MX_TRY(cudaStreamWaitEvent(cs->h2d, cs->consumed_dy[i], 0));
        MX_TRY(copy_in(c[i].dyd, t.dy, t.M, t.N, cs->h2d));
        MX_TRY(cudaEventRecord(ev_dy(i), cs->h2d));
    }
    MX_TRY(cudaEventRecord(ev_h2d_done, cs->h2d));

    // Forwards.
    for (int i = 0; i < count; ++i) {
        const mxfp4_linear_host_task& t = tasks[i];
        const Carve& b = c[i];
        const int64_t ldk = round8(t.K);
        MX_TRY(cudaStreamWaitEvent(comp, ev_xw(i), 0));
        const mxfp4_quantize_task q[2] = {
            {b.xd, t.M, t.K, ldk, b.xrq, b.xrs, b.xcq, b.xcs, 0, 0},
            {b.wd, t.N, t.K, ldk, b.wrq, b.wrs, b.wcq, b.wcs, 0, 0},
        };
        MX_TRY_ST(mxfp4_quantize_batch(2, q, t.train, MXFP4_SCALE_TC, stream));
        MX_TRY(cudaEventRecord(cs->consumed_xw[i], comp));
        MX_TRY_ST(mxfp4_gemm(b.xrq, b.xrs, b.wrq, b.wrs, t.M, t.N, t.K, b.y, t.N, t.out_dtype, stream));
        MX_TRY(cudaEventRecord(ev_y(i), comp));
        MX_TRY(cudaStreamWaitEvent(cs->d2h, ev_y(i), 0));
        MX_TRY(copy_out(t.y, b.y, t.M, t.N, t.out_dtype == MXFP4_OUT_F32 ? 4 : 2, cs->d2h));
    }
    // Backwards, last linear first.
    for (int i = count - 1; i >= 0; --i) {
        const mxfp4_linear_host_task& t = tasks[i];
        if (!t.train) continue;
        const Carve& b = c[i];
        MX_TRY(cudaStreamWaitEvent(comp, ev_dy(i), 0));
        MX_TRY_ST(mxfp4_quantize_dual(b.dyd, t.M, t.N, round8(t.N), b.drq, b.drs, b.dcq, b.dcs, MXFP4_SCALE_TC,
                                      stream));
        MX_TRY(cudaEventRecord(cs->consumed_dy[i], comp));
        const mxfp4_gemm_task g[2] = {
            {b.drq, b.drs, b.wcq, b.wcs, t.M, t.K, t.N, b.dx, t.K, t.out_dtype, nullptr},
            {b.dcq, b.dcs, b.xcq, b.xcs, t.N, t.K, t.M, b.dw, t.K, t.out_dtype, nullptr},
        };
        MX_TRY_ST(mxfp4_gemm_batch(2, g, stream));
        MX_TRY(cudaEventRecord(ev_bwd(i), comp));
        MX_TRY(cudaStreamWaitEvent(cs->d2h, ev_bwd(i), 0));
        const size_t es = t.out_dtype == MXFP4_OUT_F32 ? 4 : 2;
        MX_TRY(copy_out(t.dw, b.dw, t.N, t.K, es, cs->d2h));
        MX_TRY(copy_out(t.dx, b.dx, t.M, t.K, es, cs->d2h));
    }
    MX_TRY(cudaEventRecord(ev_d2h_done, cs->d2h));
    MX_TRY(cudaStreamWaitEvent(comp, ev_h2d_done, 0));
    if (pipelined) {
        // The caller's stream runs on; the next step writes the other output set.
        MX_TRY(cudaEventRecord(cs->slot_free[slot], cs->d2h));
        cs->slot_valid[slot] = true;
        cs->slot = slot ^ 1;
        cs->consumed_valid = true;
    } else {
        // The caller's stream is ordered after every copy of the step, so nothing of it is
        // in flight when the next step starts.
        MX_TRY(cudaStreamWaitEvent(comp, ev_d2h_done, 0));
        cs->slot_valid[0] = cs->slot_valid[1] = false;
        cs->slot = 0;
        cs->consumed_valid = false;
    }
    return MXFP4_OK;
}


}  // namespace

extern "C" {

mxfp4_status mxfp4_linear_workspace_bytes(int32_t count, const mxfp4_linear_host_task* tasks, size_t* bytes) {
    MX_TRY_ST(check_tasks(count, tasks, false));
    if (bytes == nullptr) return MXFP4_ERR_INVALID_ARG;
    *bytes = total_bytes(count, tasks);
    return MXFP4_OK;
}

mxfp4_status mxfp4_linear_step_host(int32_t count, const mxfp4_linear_host_task* tasks, void* workspace,
                                    size_t workspace_bytes, mxfp4_stream_t stream) {
    return step_host(count, tasks, workspace, workspace_bytes, stream, false);
}

mxfp4_status mxfp4_linear_pipelined_workspace_bytes(int32_t count, const mxfp4_linear_host_task* tasks,
                                                    size_t* bytes) {
    MX_TRY_ST(check_tasks(count, tasks, false));
    if (bytes == nullptr) return MXFP4_ERR_INVALID_ARG;
    *bytes = pipelined_bytes(count, tasks);
    return MXFP4_OK;
}

mxfp4_status mxfp4_linear_step_host_pipelined(int32_t count, const mxfp4_linear_host_task* tasks,
                                              void* workspace, size_t workspace_bytes, mxfp4_stream_t stream) {
    return step_host(count, tasks, workspace, workspace_bytes, stream, true);
}

mxfp4_status mxfp4_linear_host_wait(mxfp4_stream_t stream) {
    std::lock_guard<std::mutex> lock(g_host_mutex);
    CopyStreams* cs = nullptr;
    MX_TRY_ST(copy_streams(&cs));
    cudaStream_t comp = reinterpret_cast<cudaStream_t>(stream);
    MX_TRY(cudaStreamWaitEvent(comp, cs->ev[kEventsPerStep - 2], 0));
    MX_TRY(cudaStreamWaitEvent(comp, cs->ev[kEventsPerStep - 1], 0));
    return MXFP4_OK;
}

}  // extern "C"
