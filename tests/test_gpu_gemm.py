"""GPU parity of the block-scaled MXF4 GEMM (fwd, dgrad, wgrad) against the fp64 oracle.

The GPU path quantizes bf16 inputs with its own kernels and multiplies on the tensor
cores; the oracle quantizes the same bf16 inputs on the CPU and sums dequantized products
in fp64.  Accuracy contract: see tests/parity.py.
"""
import numpy as np
import pytest
import torch

import oracle
from mxfp4_block_scaled_quantize_gb300 import abi, workloads
from mxfp4_block_scaled_quantize_gb300.linear import MXFP4Linear
from parity import check_gemm, check_gemm_bias

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield
    assert abi.mxfp4_last_device_error() == abi.MXFP4_OK


def pitched(x_cpu):
    """CUDA copy of x with a row pitch rounded up to a multiple of 8 elements."""
    M, K = x_cpu.shape
    ld = (K + 7) // 8 * 8
    wide = torch.zeros((M, ld), dtype=x_cpu.dtype, device="cuda")
    wide[:, :K] = x_cpu.cuda()
    return wide[:, :K]


def gpu_gemm_from_bf16(a_cpu, b_cpu, out_dtype, ldc=None):
    """Quantize A[M,K], B[N,K] (row blobs) on the GPU and return C = A.B^T."""
    M, K = a_cpu.shape
    N = b_cpu.shape[0]
    aq, a_s = abi.quantize(pitched(a_cpu), dual=False)
    bq, b_s = abi.quantize(pitched(b_cpu), dual=False)
    ldc = ldc or N
    out = torch.full((M, ldc), float("nan"), dtype=out_dtype, device="cuda")
    abi.mxfp4_gemm(aq, a_s, bq, b_s, M, N, K, out, ldc,
                   abi.MXFP4_OUT_F32 if out_dtype == torch.float32 else abi.MXFP4_OUT_BF16)
    torch.cuda.synchronize()
    assert abi.mxfp4_last_device_error() == abi.MXFP4_OK
    return out


def oracle_gemm_from_bf16(a_cpu, b_cpu, rows=None):
    ab, bb = workloads.bf16_bits(a_cpu), workloads.bf16_bits(b_cpu)
    if rows is not None:
        ab = np.ascontiguousarray(ab[rows])
    aq, a_s = oracle.quantize_row(ab)
    bq, b_s = oracle.quantize_row(bb)
    return oracle.gemm(aq, a_s, bq, b_s)


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_tiny_config_step(out_dtype):
    wl = workloads.TINY
    lin = wl.linears[0]
    t = wl.tensors(0)
    layer = MXFP4Linear(lin.M, lin.N, lin.K, train=True, out_dtype=out_dtype)
    y, dx, dw = layer.step(t["X"].cuda(), t["W"].cuda(), t["dY"].cuda())
    torch.cuda.synchronize()
    assert abi.mxfp4_last_device_error() == abi.MXFP4_OK
    X, W, DY = (oracle.quantize_dual(workloads.bf16_bits(t[k])) for k in ("X", "W", "dY"))
    c, cabs = oracle.gemm(X[0], X[1], W[0], W[1])
    check_gemm(y, c, cabs, "tiny fwd")
    c, cabs = oracle.gemm(DY[0], DY[1], W[2], W[3])
    check_gemm(dx, c, cabs, "tiny dgrad")
    c, cabs = oracle.gemm(DY[2], DY[3], X[2], X[3])
    check_gemm(dw, c, cabs, "tiny wgrad")


def test_step_from_host_matches_device_step():
    # The overlapped host-buffer step (copy streams + kernel stream) gives the same bytes as
    # the plain device step, twice in a row (buffers reused across steps).
    lin = workloads.Linear("host", 384, 640, 512, True)
    wl = workloads.Workload("host", "host-buffer step", [lin], base_seed=11)
    t = wl.tensors(0)
    ref = MXFP4Linear(lin.M, lin.N, lin.K, train=True)
    want = [o.cpu() for o in ref.step(t["X"].cuda(), t["W"].cuda(), t["dY"].cuda())]
    layer = MXFP4Linear(lin.M, lin.N, lin.K, train=True)
    hx, hw, hdy = (t[k].pin_memory() for k in ("X", "W", "dY"))
    for _ in range(2):
        outs = [torch.full(o.shape, float("nan"), dtype=o.dtype).pin_memory() for o in want]
        layer.step_host(hx, hw, hdy, *outs)
        torch.cuda.synchronize()
        assert abi.mxfp4_last_device_error() == abi.MXFP4_OK
        for got, exp in zip(outs, want):
            assert torch.equal(got.view(torch.int16), exp.view(torch.int16))


def test_block_host_step_matches_device_step():
    # The library's host-buffer step (mxfp4_linear_step_host) over three linears -- two
    # training, one forward-only; bf16 and fp32 outputs; K = 1001 needs a pitched device copy
    # -- gives the bytes of the device step of each linear, twice in a row (workspace and
    # copy streams reused).
    from mxfp4_block_scaled_quantize_gb300.linear import MXFP4Block
    shapes = [("a", 300, 520, 200, True, torch.bfloat16), ("b", 257, 136, 1001, True, torch.float32),
              ("c", 130, 264, 384, False, torch.bfloat16)]
    host_in, want = [], []
    for i, (_, M, N, K, train, od) in enumerate(shapes):
        t = {"X": workloads.student_t3((M, K), 1.0, 71 + i), "W": workloads.normal((N, K), 0.3, 81 + i)}
        if train:
            t["dY"] = workloads.normal((M, N), 0.01, 91 + i)
        host_in.append({k: v.pin_memory() for k, v in t.items()})
        ref = MXFP4Linear(M, N, K, train=train, out_dtype=od)
        outs = ref.step(pitched(t["X"]), pitched(t["W"]), pitched(t["dY"]) if train else None)
        want.append([o.cpu() for o in outs])
    torch.cuda.synchronize()
    tasks = []
    for (_, M, N, K, train, od), hi in zip(shapes, host_in):
        code = abi.MXFP4_OUT_F32 if od == torch.float32 else abi.MXFP4_OUT_BF16
        tasks.append([hi["X"], hi["W"], hi.get("dY"), None, None, None, M, N, K, train, code])
    need = abi.mxfp4_linear_workspace_bytes(tasks)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    for _ in range(2):
        got = []
        for tk, w_ in zip(tasks, want):
            outs = [torch.full(o.shape, float("nan"), dtype=o.dtype).pin_memory() for o in w_]
            tk[3:3 + len(outs)] = outs
            got.append(outs)
        abi.mxfp4_linear_step_host([tuple(t) for t in tasks], ws, need)
        torch.cuda.current_stream().synchronize()
        assert abi.mxfp4_last_device_error() == abi.MXFP4_OK
        for g_, w_ in zip(got, want):
            for a, b in zip(g_, w_):
                assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))


def test_pipelined_host_steps_match_device_steps():
    # Five consecutive host-buffer steps of two linears (one training with bf16 outputs, one
    # forward-only with fp32 outputs), each step with inputs of its own: four through the
    # pipelined entry point (the two output sets each used twice, the inputs refilled while
    # the previous step's results are still being copied out) and a plain call in the middle.
    # Every step's host results are the bytes of the device step on that step's inputs.
    shapes = [(300, 520, 200, True, torch.bfloat16), (257, 136, 1001, False, torch.float32)]
    steps = 5
    host_in, want = [], []
    for k in range(steps):
        hin, wk = [], []
        for i, (M, N, K, train, od) in enumerate(shapes):
            t = {"X": workloads.student_t3((M, K), 1.0, 1000 + 10 * k + i),
                 "W": workloads.normal((N, K), 0.3, 2000 + 10 * k + i)}
            if train:
                t["dY"] = workloads.normal((M, N), 0.01, 3000 + 10 * k + i)
            hin.append({n: v.pin_memory() for n, v in t.items()})
            ref = MXFP4Linear(M, N, K, train=train, out_dtype=od)
            outs = ref.step(pitched(t["X"]), pitched(t["W"]), pitched(t["dY"]) if train else None)
            wk.append([o.cpu() for o in outs])
        host_in.append(hin)
        want.append(wk)
    torch.cuda.synchronize()
    got = []
    tasks_of = []
    for k in range(steps):
        tasks, gk = [], []
        for (M, N, K, train, od), hi, w_ in zip(shapes, host_in[k], want[k]):
            code = abi.MXFP4_OUT_F32 if od == torch.float32 else abi.MXFP4_OUT_BF16
            outs = [torch.full(o.shape, float("nan"), dtype=o.dtype).pin_memory() for o in w_]
            outs3 = outs + [None] * (3 - len(outs))
            tasks.append((hi["X"], hi["W"], hi.get("dY"), *outs3, M, N, K, train, code))
            gk.append(outs)
        tasks_of.append(tasks)
        got.append(gk)
    need = abi.mxfp4_linear_pipelined_workspace_bytes(tasks_of[0])
    assert need > abi.mxfp4_linear_workspace_bytes(tasks_of[0])
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    for k in range(steps):
        if k == 2:
            abi.mxfp4_linear_step_host(tasks_of[k], ws, need)
        else:
            abi.mxfp4_linear_step_host_pipelined(tasks_of[k], ws, need)
    abi.mxfp4_linear_host_wait()
    torch.cuda.current_stream().synchronize()
    assert abi.mxfp4_last_device_error() == abi.MXFP4_OK
    for k in range(steps):
        for g_, w_ in zip(got[k], want[k]):
            for a, b in zip(g_, w_):
                assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), f"step {k}"


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (1, 8, 32), (200, 300, 40), (129, 257, 384),
                                   (128, 256, 256), (300, 520, 1000), (64, 1000, 4600),
                                   (256, 128, 128), (384, 768, 640), (513, 255, 2048)])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_ragged_shapes(M, N, K, out_dtype):
    a = workloads.student_t3((M, K), 1.0, M + 3 * N + 7 * K)
    b = workloads.normal((N, K), 0.5, M + 5 * N + 11 * K)
    c_gpu = gpu_gemm_from_bf16(a, b, out_dtype)
    c, cabs = oracle_gemm_from_bf16(a, b)
    check_gemm(c_gpu, c, cabs, f"gemm {M}x{N}x{K}")


def bias_bf16(N, seed):
    """A bf16 bias vector with magnitudes spread over 2^-8 .. 2^8 (as uint16 bits and a
    CUDA tensor)."""
    rng = np.random.default_rng(seed)
    v = rng.standard_normal(N) * np.ldexp(1.0, rng.integers(-8, 9, N))
    bits = oracle.round_to_bf16(v)
    t = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
    return bits, t


@pytest.mark.parametrize("M,N,K", [(1, 8, 32), (200, 300, 40), (129, 257, 384), (64, 1000, 4600),
                                   (384, 768, 640), (513, 255, 2048)])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_gemm_bias(M, N, K, out_dtype):
    # The fused `output + bias` against the oracle's GEMM followed by its bias add; N not a
    # multiple of 8 exercises the bias reads at the ragged right edge.
    a = workloads.student_t3((M, K), 1.0, 31 + M + 3 * N + 7 * K)
    b = workloads.normal((N, K), 0.5, 37 + M + 5 * N + 11 * K)
    bits, bias = bias_bf16(N, M + N + K)
    aq, a_s = abi.quantize(pitched(a), dual=False)
    bq, b_s = abi.quantize(pitched(b), dual=False)
    out = abi.gemm(aq, a_s, bq, b_s, M, N, K, out_dtype=out_dtype, bias=bias)
    torch.cuda.synchronize()
    assert abi.mxfp4_last_device_error() == abi.MXFP4_OK
    c, cabs = oracle_gemm_from_bf16(a, b)
    check_gemm_bias(out, c, cabs, bits, f"gemm+bias {M}x{N}x{K}")


def test_flux_mlp_forward_bias_sampled():
    # Full Flux-12B MLP up-projection forward (M 4608, N 12288, K 3072) with the layer's
    # bias, in the launch configuration of the forward step; sampled output rows.
    wl = workloads.FLUX_MLP_STEP
    lin = wl.linears[0]
    t = wl.tensors(0)
    bits, bias = bias_bf16(lin.N, 7)
    layer = MXFP4Linear(lin.M, lin.N, lin.K, train=False)
    layer.quantize_xw(t["X"].cuda(), t["W"].cuda())
    y = layer.fwd_gemm(bias=bias)
    torch.cuda.synchronize()
    assert abi.mxfp4_last_device_error() == abi.MXFP4_OK
    rows = np.array([0, 1, 127, 128, 255, 256, 2047, 3333, 4480, 4607])
    c, cabs = oracle_gemm_from_bf16(t["X"], t["W"], rows=rows)
    check_gemm_bias(y[torch.as_tensor(rows, device="cuda")], c, cabs, bits, "flux mlp fwd + bias")


def test_batch_with_bias_equals_single_calls():
    # Batched problems with and without a bias give each problem its own call's bytes.
    probs = [(384, 768, 640, torch.bfloat16, True), (129, 257, 384, torch.float32, True),
             (513, 255, 2048, torch.float32, False), (256, 520, 1000, torch.bfloat16, True)]
    tasks, outs, refs = [], [], []
    for i, (M, N, K, od, with_bias) in enumerate(probs):
        a = workloads.student_t3((M, K), 1.0, 301 + i)
        b = workloads.normal((N, K), 0.5, 401 + i)
        aq, a_s = abi.quantize(pitched(a), dual=False)
        bq, b_s = abi.quantize(pitched(b), dual=False)
        code = abi.MXFP4_OUT_F32 if od == torch.float32 else abi.MXFP4_OUT_BF16
        bias = bias_bf16(N, 501 + i)[1] if with_bias else None
        ref = torch.full((M, N), float("nan"), dtype=od, device="cuda")
        if with_bias:
            abi.mxfp4_gemm_bias(aq, a_s, bq, b_s, M, N, K, bias, ref, N, code)
        else:
            abi.mxfp4_gemm(aq, a_s, bq, b_s, M, N, K, ref, N, code)
        out = torch.full((M, N), float("nan"), dtype=od, device="cuda")
        tasks.append((aq, a_s, bq, b_s, M, N, K, out, N, code, bias))
        outs.append(out)
        refs.append(ref)
    abi.mxfp4_gemm_batch(tasks)
    torch.cuda.synchronize()
    assert abi.mxfp4_last_device_error() == abi.MXFP4_OK
    for out, ref in zip(outs, refs):
        assert torch.equal(out.view(torch.uint8).cpu(), ref.view(torch.uint8).cpu())


def test_batch_equals_single_calls():
    # One batched call over 1..4 problems (CTA-pair and one-CTA shapes, ragged edges, bf16
    # and fp32 outputs, a pitched output) gives each problem exactly its own call's bytes.
    probs = [(384, 768, 640, torch.bfloat16, 768), (129, 257, 384, torch.float32, 260),
             (64, 1000, 4600, torch.bfloat16, 1000), (513, 255, 2048, torch.float32, 256)]
    ins, singles = [], []
    for i, (M, N, K, od, ldc) in enumerate(probs):
        a = workloads.student_t3((M, K), 1.0, 101 + i)
        b = workloads.normal((N, K), 0.5, 201 + i)
        aq, a_s = abi.quantize(pitched(a), dual=False)
        bq, b_s = abi.quantize(pitched(b), dual=False)
        code = abi.MXFP4_OUT_F32 if od == torch.float32 else abi.MXFP4_OUT_BF16
        ins.append((aq, a_s, bq, b_s, M, N, K, code))
        ref = torch.full((M, ldc), float("nan"), dtype=od, device="cuda")
        abi.mxfp4_gemm(aq, a_s, bq, b_s, M, N, K, ref, ldc, code)
        singles.append(ref)
    torch.cuda.synchronize()
    for n in (1, 2, 4):
        outs, tasks = [], []
        for (aq, a_s, bq, b_s, M, N, K, code), ref in zip(ins[:n], singles[:n]):
            out = torch.full(ref.shape, float("nan"), dtype=ref.dtype, device="cuda")
            tasks.append((aq, a_s, bq, b_s, M, N, K, out, out.stride(0), code))
            outs.append(out)
        abi.mxfp4_gemm_batch(tasks)
        torch.cuda.synchronize()
        assert abi.mxfp4_last_device_error() == abi.MXFP4_OK
        for out, ref in zip(outs, singles):
            # byte-identical, the pitch tail (never written) included
            assert torch.equal(out.view(torch.uint8).cpu(), ref.view(torch.uint8).cpu())


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_output_pitch_and_untouched_tail(out_dtype):
    M, N, K = 200, 300, 512
    a = workloads.normal((M, K), 1.0, 1)
    b = workloads.normal((N, K), 1.0, 2)
    ldc = N + 13                      # odd pitch: no vector stores possible
    out = gpu_gemm_from_bf16(a, b, out_dtype, ldc=ldc)
    assert torch.all(torch.isnan(out[:, N:].float()))   # columns past N untouched
    c, cabs = oracle_gemm_from_bf16(a, b)
    check_gemm(out[:, :N], c, cabs, "gemm ldc=N+13")


def _sample_rows(M, n=12, seed=0):
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([rng.choice(M, n, replace=False), [0, M - 1]]))


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_flux_qkv_forward_sampled(out_dtype):
    wl = workloads.FLUX_QKV_FWD
    lin = wl.linears[0]
    t = wl.tensors(0)
    layer = MXFP4Linear(lin.M, lin.N, lin.K, train=False, out_dtype=out_dtype)
    (y,) = layer.step(t["X"].cuda(), t["W"].cuda())
    torch.cuda.synchronize()
    assert abi.mxfp4_last_device_error() == abi.MXFP4_OK
    rows = _sample_rows(lin.M)
    c, cabs = oracle_gemm_from_bf16(t["X"], t["W"], rows)
    check_gemm(y[torch.as_tensor(rows, device="cuda")], c, cabs, "flux qkv fwd")


def test_flux_mlp_training_step_sampled():
    wl = workloads.FLUX_MLP_STEP
    lin = wl.linears[0]
    t = wl.tensors(0)
    layer = MXFP4Linear(lin.M, lin.N, lin.K, train=True)
    y, dx, dw = layer.step(t["X"].cuda(), t["W"].cuda(), t["dY"].cuda())
    torch.cuda.synchronize()
    assert abi.mxfp4_last_device_error() == abi.MXFP4_OK
    xb, wb, dyb = (workloads.bf16_bits(t[k]) for k in ("X", "W", "dY"))
    rows = _sample_rows(lin.M, 8, 1)
    # fwd: rows of Y need X rows and all of W's row blob
    aq, a_s = oracle.quantize_row(np.ascontiguousarray(xb[rows]))
    wq, ws = oracle.quantize_row(wb)
    c, cabs = oracle.gemm(aq, a_s, wq, ws)
    check_gemm(y[torch.as_tensor(rows, device="cuda")], c, cabs, "mlp fwd")
    # dgrad: rows of dX need dY rows and all of W's col blob
    aq, a_s = oracle.quantize_row(np.ascontiguousarray(dyb[rows]))
    wcq, wcs = oracle.quantize_col(wb)
    c, cabs = oracle.gemm(aq, a_s, wcq, wcs)
    check_gemm(dx[torch.as_tensor(rows, device="cuda")], c, cabs, "mlp dgrad")
    # wgrad: rows n of dW need column n of dY (its col-blob row) and all of X's col blob
    nrows = _sample_rows(lin.N, 8, 2)
    aq, a_s = oracle.quantize_col(np.ascontiguousarray(dyb[:, nrows]))
    xcq, xcs = oracle.quantize_col(xb)
    c, cabs = oracle.gemm(aq, a_s, xcq, xcs)
    check_gemm(dw[torch.as_tensor(nrows, device="cuda")], c, cabs, "mlp wgrad")


def test_flux_linear2_forward_long_k_sampled():
    lin = workloads.FLUX_SINGLE_BLOCK.linears[1]          # K = 15360
    t = workloads.FLUX_SINGLE_BLOCK.tensors(1)
    c_gpu = gpu_gemm_from_bf16(t["X"], t["W"], torch.bfloat16)
    rows = _sample_rows(lin.M, 6, 3)
    c, cabs = oracle_gemm_from_bf16(t["X"], t["W"], rows)
    check_gemm(c_gpu[torch.as_tensor(rows, device="cuda")], c, cabs, "linear2 fwd")


def test_gemm_argument_errors():
    lib = abi.load()
    q, s = abi.alloc_blob(128, 128)
    c = torch.empty((128, 128), dtype=torch.bfloat16, device="cuda")
    p = lambda t: t.data_ptr()
    assert lib.mxfp4_gemm(p(q), p(s), p(q), p(s), 128, 128, 128, p(c), 64, 0, None) == abi.MXFP4_ERR_INVALID_ARG
    assert lib.mxfp4_gemm(p(q), p(s), p(q), p(s), 128, 128, 0, p(c), 128, 0, None) == abi.MXFP4_ERR_INVALID_ARG
    assert lib.mxfp4_gemm(p(q) + 8, p(s), p(q), p(s), 128, 128, 128, p(c), 128, 0, None) == abi.MXFP4_ERR_MISALIGNED
    assert lib.mxfp4_gemm(p(q), p(s), p(q), p(s), 128, 128, 128, p(c), 128, 5, None) == abi.MXFP4_ERR_INVALID_ARG


@pytest.mark.parametrize("backward", ["mxfp4", "fp8"])
def test_repeated_steps_are_bit_identical(backward):
    # The same kernels with the same arguments give bit-identical outputs: every output tile
    # is computed by one CTA pair in a fixed K order, and the only atomic (the FP8 amax) is
    # a maximum, which does not depend on the order of arrival.
    wl = workloads.FLUX_MLP_STEP
    lin = wl.linears[0]
    t = wl.tensors(0)
    x, w, dy = (t[k].cuda() for k in ("X", "W", "dY"))
    layer = MXFP4Linear(lin.M, lin.N, lin.K, train=True, backward=backward)
    first = [o.clone() for o in layer.step(x, w, dy)]
    for _ in range(2):
        outs = layer.step(x, w, dy)
        torch.cuda.synchronize()
        for a, b in zip(outs, first):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert abi.mxfp4_last_device_error() == abi.MXFP4_OK


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_tiny_step_with_2d_weight_blocks(out_dtype):
    # The layer with the weight recipe (32 x 32 blocks for W in both packings): forward and
    # dgrad read W's 2-D blobs, wgrad is unchanged; every GEMM against the oracle's GEMM over
    # the oracle's 2-D blobs.
    wl = workloads.TINY
    lin = wl.linears[0]
    t = wl.tensors(0)
    layer = MXFP4Linear(lin.M, lin.N, lin.K, train=True, out_dtype=out_dtype, weight_2d=True)
    y, dx, dw = layer.step(t["X"].cuda(), t["W"].cuda(), t["dY"].cuda())
    torch.cuda.synchronize()
    assert abi.mxfp4_last_device_error() == abi.MXFP4_OK
    xb, wb, dyb = (workloads.bf16_bits(t[k]) for k in ("X", "W", "dY"))
    X, DY = oracle.quantize_dual(xb), oracle.quantize_dual(dyb)
    wr, wc = oracle.quantize_row_2d(wb), oracle.quantize_col_2d(wb)
    c, cabs = oracle.gemm(X[0], X[1], *wr)
    check_gemm(y, c, cabs, "tiny fwd, 2-D W")
    c, cabs = oracle.gemm(DY[0], DY[1], *wc)
    check_gemm(dx, c, cabs, "tiny dgrad, 2-D W")
    c, cabs = oracle.gemm(DY[2], DY[3], X[2], X[3])
    check_gemm(dw, c, cabs, "tiny wgrad")


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("shape,sr_seed", [((256, 256, 512), None), ((200, 136, 264), None),
                                           ((256, 256, 512), 31), ((200, 136, 264), 2**40 + 1)])
def test_step_with_both_recipes(shape, sr_seed, out_dtype):
    # The layer with the pages' recipes: W in 32 x 32 blocks, the col blobs of X and dY
    # transformed (the same signs), and with a seed dY stochastically rounded (the gradient
    # recipe with `use_sr`).  fwd and dgrad read W's 2-D blobs; wgrad multiplies the two
    # transformed col blobs.  Every GEMM against the oracle's GEMM over the oracle's blobs
    # of the same recipes.
    M, N, K = shape
    t = {"X": workloads.student_t3((M, K), 1.0, M + 1), "W": workloads.normal((N, K), 0.3, N + 2),
         "dY": workloads.normal((M, N), 0.01, K + 3)}
    layer = MXFP4Linear(M, N, K, train=True, out_dtype=out_dtype, weight_2d=True, rht_signs=0xA5C3)
    y, dx, dw = layer.step(pitched(t["X"]), pitched(t["W"]), pitched(t["dY"]), sr_seed=sr_seed)
    torch.cuda.synchronize()
    assert abi.mxfp4_last_device_error() == abi.MXFP4_OK
    xb, wb, dyb = (workloads.bf16_bits(t[k]) for k in ("X", "W", "dY"))
    xr = oracle.quantize_row(xb)
    wr, wc = oracle.quantize_row_2d(wb), oracle.quantize_col_2d(wb)
    xc = oracle.quantize_col_rht(xb, 0xA5C3)
    if sr_seed is None:
        dyr, dyc = oracle.quantize_row(dyb), oracle.quantize_col_rht(dyb, 0xA5C3)
    else:
        dyr, dyc = oracle.quantize_row_sr(dyb, sr_seed), oracle.quantize_col_rht_sr(dyb, 0xA5C3, sr_seed)
    c, cabs = oracle.gemm(*xr, *wr)
    check_gemm(y, c, cabs, f"recipes fwd {shape}")
    c, cabs = oracle.gemm(*dyr, *wc)
    check_gemm(dx, c, cabs, f"recipes dgrad {shape}")
    c, cabs = oracle.gemm(*dyc, *xc)
    check_gemm(dw, c, cabs, f"recipes wgrad {shape}")


@pytest.fixture
def tile_policy():
    """Set the CTA-pair tile width for one test; AUTO again afterwards."""
    yield abi.mxfp4_gemm_set_tile_policy
    abi.mxfp4_gemm_set_tile_policy(abi.MXFP4_TILES_AUTO)


@pytest.mark.parametrize("M,N,K", [(384, 768, 640), (300, 520, 1000), (513, 1000, 2048), (257, 385, 128),
                                   (1000, 1152, 384), (640, 2304, 4608), (2048, 383, 256),
                                   (6500, 520, 256), (256, 384, 256), (300, 64, 256), (1024, 136, 512),
                                   (129, 392, 96)])
def test_wide_tiles_match_oracle_and_narrow_tiles(M, N, K, tile_policy):
    # 256 x 384 tiles (one N 256 and one N 128 MMA per K slice, ragged M, N and K edges,
    # tile grids of one to several waves) against the oracle, and bit for bit against the
    # 256 x 256 tiles.  M 6500 has 26 row tiles: its tiles are walked in groups of 8 row
    # tiles, the last group holding 2.  N 64 and 136 leave the N 128 MMA's rows (and part of
    # the N 256 one's) wholly past N; M 129 leaves the odd CTA one row, K 96 one scale atom.
    a = workloads.student_t3((M, K), 1.0, 11 + M + 3 * N + 7 * K)
    b = workloads.normal((N, K), 0.5, 13 + M + 5 * N + 11 * K)
    tile_policy(abi.MXFP4_TILES_WIDE)
    wide = gpu_gemm_from_bf16(a, b, torch.bfloat16)
    tile_policy(abi.MXFP4_TILES_NARROW)
    narrow = gpu_gemm_from_bf16(a, b, torch.bfloat16)
    c, cabs = oracle_gemm_from_bf16(a, b)
    check_gemm(wide, c, cabs, f"wide gemm {M}x{N}x{K}")
    assert torch.equal(wide.view(torch.uint8).cpu(), narrow.view(torch.uint8).cpu())


@pytest.mark.parametrize("M,N,K", [(384, 768, 640), (513, 1000, 2048)])
def test_wide_tiles_with_bias(M, N, K, tile_policy):
    a = workloads.student_t3((M, K), 1.0, 41 + M + 3 * N + 7 * K)
    b = workloads.normal((N, K), 0.5, 43 + M + 5 * N + 11 * K)
    bits, bias = bias_bf16(N, 47 + M + N + K)
    aq, a_s = abi.quantize(pitched(a), dual=False)
    bq, b_s = abi.quantize(pitched(b), dual=False)
    tile_policy(abi.MXFP4_TILES_WIDE)
    out = abi.gemm(aq, a_s, bq, b_s, M, N, K, out_dtype=torch.bfloat16, bias=bias)
    torch.cuda.synchronize()
    assert abi.mxfp4_last_device_error() == abi.MXFP4_OK
    c, cabs = oracle_gemm_from_bf16(a, b)
    check_gemm_bias(out, c, cabs, bits, f"wide gemm+bias {M}x{N}x{K}")


def test_wide_policy_batch_equals_narrow_singles(tile_policy):
    # A batch under the wide policy (bf16 pair problems, a one-CTA problem beside them, a
    # pitched output) gives each problem the bytes of its own narrow call; a batch holding an
    # fp32 pair problem runs narrow tiles and gives the same bytes too.
    probs = [(384, 768, 640, torch.bfloat16, 776), (513, 1000, 2048, torch.bfloat16, 1000),
             (64, 1000, 4600, torch.bfloat16, 1000), (300, 520, 1000, torch.float32, 520)]
    ins, singles = [], []
    tile_policy(abi.MXFP4_TILES_NARROW)
    for i, (M, N, K, od, ldc) in enumerate(probs):
        a = workloads.student_t3((M, K), 1.0, 601 + i)
        b = workloads.normal((N, K), 0.5, 701 + i)
        aq, a_s = abi.quantize(pitched(a), dual=False)
        bq, b_s = abi.quantize(pitched(b), dual=False)
        code = abi.MXFP4_OUT_F32 if od == torch.float32 else abi.MXFP4_OUT_BF16
        ins.append((aq, a_s, bq, b_s, M, N, K, code))
        ref = torch.full((M, ldc), float("nan"), dtype=od, device="cuda")
        abi.mxfp4_gemm(aq, a_s, bq, b_s, M, N, K, ref, ldc, code)
        singles.append(ref)
    torch.cuda.synchronize()
    tile_policy(abi.MXFP4_TILES_WIDE)
    for sel in ((0, 1, 2), (0, 3)):
        outs, tasks = [], []
        for i in sel:
            aq, a_s, bq, b_s, M, N, K, code = ins[i]
            out = torch.full(singles[i].shape, float("nan"), dtype=singles[i].dtype, device="cuda")
            tasks.append((aq, a_s, bq, b_s, M, N, K, out, out.stride(0), code))
            outs.append(out)
        abi.mxfp4_gemm_batch(tasks)
        torch.cuda.synchronize()
        assert abi.mxfp4_last_device_error() == abi.MXFP4_OK
        for i, out in zip(sel, outs):
            assert torch.equal(out.view(torch.uint8).cpu(), singles[i].view(torch.uint8).cpu())


def test_flux_linear1_step_wide_tiles_sampled(tile_policy):
    # The single-stream block's linear1 training step at full size on 256 x 384 tiles: the
    # forward 4608 x 21504 x 3072, and dgrad 4608 x 3072 x 21504 with wgrad 21504 x 3072 x
    # 4608 in one launch, as the step runs them; sampled rows against the oracle.
    wl = workloads.FLUX_SINGLE_BLOCK
    lin = wl.linears[0]
    t = wl.tensors(0)
    tile_policy(abi.MXFP4_TILES_WIDE)
    layer = MXFP4Linear(lin.M, lin.N, lin.K, train=True)
    y, dx, dw = layer.step(t["X"].cuda(), t["W"].cuda(), t["dY"].cuda())
    torch.cuda.synchronize()
    assert abi.mxfp4_last_device_error() == abi.MXFP4_OK
    xb, wb, dyb = (workloads.bf16_bits(t[k]) for k in ("X", "W", "dY"))
    rows = _sample_rows(lin.M, 6, 3)
    aq, a_s = oracle.quantize_row(np.ascontiguousarray(xb[rows]))
    wq, ws = oracle.quantize_row(wb)
    c, cabs = oracle.gemm(aq, a_s, wq, ws)
    check_gemm(y[torch.as_tensor(rows, device="cuda")], c, cabs, "linear1 fwd (wide)")
    aq, a_s = oracle.quantize_row(np.ascontiguousarray(dyb[rows]))
    wcq, wcs = oracle.quantize_col(wb)
    c, cabs = oracle.gemm(aq, a_s, wcq, wcs)
    check_gemm(dx[torch.as_tensor(rows, device="cuda")], c, cabs, "linear1 dgrad (wide)")
    nrows = _sample_rows(lin.N, 6, 4)
    aq, a_s = oracle.quantize_col(np.ascontiguousarray(dyb[:, nrows]))
    xcq, xcs = oracle.quantize_col(xb)
    c, cabs = oracle.gemm(aq, a_s, xcq, xcs)
    check_gemm(dw[torch.as_tensor(nrows, device="cuda")], c, cabs, "linear1 wgrad (wide)")


def test_wide_batch_with_bias_equals_narrow_singles(tile_policy):
    # The batched wide instance with a bias (two bf16 CTA-pair problems, one with a bias and
    # one without) gives each problem the bytes of its own narrow call.
    probs = [(384, 768, 640, True), (513, 1000, 2048, False), (640, 1152, 384, True)]
    tasks, outs, refs = [], [], []
    for i, (M, N, K, with_bias) in enumerate(probs):
        a = workloads.student_t3((M, K), 1.0, 801 + i)
        b = workloads.normal((N, K), 0.5, 901 + i)
        aq, a_s = abi.quantize(pitched(a), dual=False)
        bq, b_s = abi.quantize(pitched(b), dual=False)
        bias = bias_bf16(N, 1001 + i)[1] if with_bias else None
        tile_policy(abi.MXFP4_TILES_NARROW)
        ref = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        if with_bias:
            abi.mxfp4_gemm_bias(aq, a_s, bq, b_s, M, N, K, bias, ref, N, abi.MXFP4_OUT_BF16)
        else:
            abi.mxfp4_gemm(aq, a_s, bq, b_s, M, N, K, ref, N, abi.MXFP4_OUT_BF16)
        out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        tasks.append((aq, a_s, bq, b_s, M, N, K, out, N, abi.MXFP4_OUT_BF16, bias))
        outs.append(out)
        refs.append(ref)
    tile_policy(abi.MXFP4_TILES_WIDE)
    abi.mxfp4_gemm_batch(tasks)
    torch.cuda.synchronize()
    assert abi.mxfp4_last_device_error() == abi.MXFP4_OK
    for out, ref in zip(outs, refs):
        assert torch.equal(out.view(torch.uint8).cpu(), ref.view(torch.uint8).cpu())
