"""GPU parity of the hybrid FP8 backward (`backward_is_fp8` of `MXFP4LinearFunction`):
tensorwise E5M2 quantization bit for bit against the oracle (codes of both copies, amax
and scale_inv), the FP8 GEMM within the GEMM accuracy contract (tests/parity.py), and the
layer's hybrid backward step.
"""
import numpy as np
import pytest
import torch

import oracle
from mxfp4_block_scaled_quantize_gb300 import abi, workloads
from mxfp4_block_scaled_quantize_gb300.linear import MXFP4Linear
from parity import assert_bytes_equal, check_gemm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield
    assert abi.mxfp4_last_device_error() == abi.MXFP4_OK


def pitched(x_cpu):
    M, K = x_cpu.shape
    ld = (K + 7) // 8 * 8
    wide = torch.zeros((M, ld), dtype=x_cpu.dtype, device="cuda")
    wide[:, :K] = x_cpu.cuda()
    return wide[:, :K]


def f32_bits(t):
    return np.asarray(t.cpu().numpy(), np.float32).view(np.uint32)


def check_fp8_quant(x_cpu, what):
    xb = workloads.bf16_bits(x_cpu)
    qr, qc, amax, inv = abi.fp8_quantize(pitched(x_cpu))
    torch.cuda.synchronize()
    assert abi.mxfp4_last_device_error() == abi.MXFP4_OK
    oqr, oqc, oamax, oinv = oracle.fp8_quantize_tw(xb)
    assert_bytes_equal(qr.cpu().numpy(), oqr, f"{what} row codes")
    assert_bytes_equal(qc.cpu().numpy(), oqc, f"{what} col codes")
    assert f32_bits(amax)[0] == np.float32(oamax).view(np.uint32), f"{what} amax"
    assert f32_bits(inv)[0] == np.float32(oinv).view(np.uint32), f"{what} scale_inv"


@pytest.mark.parametrize("M,K", [(1, 8), (1, 40), (32, 8), (100, 40), (130, 200), (257, 33), (256, 512),
                                 (129, 129), (640, 384), (4600, 256)])
def test_fp8_quantize_ragged(M, K):
    x = workloads.inject_edge_blocks(workloads.student_t3((M, K), 1.0, 5 * M + K), 5 * M + K + 1)
    check_fp8_quant(x, f"fp8 {M}x{K}")


@pytest.mark.parametrize("scale", [1.0, 1e-3, 1e3])
def test_fp8_quantize_distributions(scale):
    check_fp8_quant(workloads.normal((384, 1000), scale, 9), f"fp8 normal x{scale}")


def test_fp8_quantize_degenerate_tensors():
    # all zero (scale 1), all the smallest subnormal (57344 / amax overflows fp32), and a
    # tensor whose amax is the largest finite bf16
    z = torch.zeros((64, 64), dtype=torch.bfloat16)
    check_fp8_quant(z, "fp8 zeros")
    tiny = torch.from_numpy(np.full((64, 48), 0x0001, np.int16)).view(torch.bfloat16)
    check_fp8_quant(tiny, "fp8 tiny")
    big = workloads.normal((64, 80), 1.0, 3).clone()
    big[5, 7] = torch.from_numpy(np.array([0x7F7F], np.int16)).view(torch.bfloat16)[0]
    check_fp8_quant(big, "fp8 near max")


def gemm_case(M, N, K, seed, out_dtype):
    a = workloads.student_t3((M, K), 1.0, seed)
    b = workloads.normal((N, K), 0.02, seed + 1)
    qa, _, _, sa = abi.fp8_quantize(pitched(a), col=False)
    qb, _, _, sb = abi.fp8_quantize(pitched(b), col=False)
    out = abi.fp8_gemm(qa, sa, qb, sb, M, N, K, out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert abi.mxfp4_last_device_error() == abi.MXFP4_OK
    oqa, _, _, osa = oracle.fp8_quantize_tw(workloads.bf16_bits(a), col=False)
    oqb, _, _, osb = oracle.fp8_quantize_tw(workloads.bf16_bits(b), col=False)
    c, cabs = oracle.fp8_gemm(oqa, osa, oqb, osb, K)
    return out, c, cabs


@pytest.mark.parametrize("M,N,K", [(1, 8, 16), (200, 300, 40), (129, 257, 384), (256, 256, 128),
                                   (300, 520, 1000), (64, 1000, 4600), (513, 255, 2048)])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_fp8_gemm_ragged(M, N, K, out_dtype):
    out, c, cabs = gemm_case(M, N, K, M + 3 * N + 7 * K, out_dtype)
    check_gemm(out, c, cabs, f"fp8 gemm {M}x{N}x{K}")


def test_fp8_batch_equals_single_calls():
    probs = [(384, 768, 640, torch.bfloat16), (129, 257, 384, torch.float32), (513, 255, 2048, torch.float32)]
    tasks, outs, refs = [], [], []
    for i, (M, N, K, od) in enumerate(probs):
        a = workloads.student_t3((M, K), 1.0, 601 + i)
        b = workloads.normal((N, K), 0.5, 701 + i)
        qa, _, _, sa = abi.fp8_quantize(pitched(a), col=False)
        qb, _, _, sb = abi.fp8_quantize(pitched(b), col=False)
        code = abi.MXFP4_OUT_F32 if od == torch.float32 else abi.MXFP4_OUT_BF16
        ref = torch.full((M, N), float("nan"), dtype=od, device="cuda")
        abi.mxfp4_fp8_gemm(qa, sa, qb, sb, M, N, K, ref, N, code)
        out = torch.full((M, N), float("nan"), dtype=od, device="cuda")
        tasks.append((qa, sa, qb, sb, M, N, K, out, N, code))
        outs.append(out)
        refs.append(ref)
    abi.mxfp4_fp8_gemm_batch(tasks)
    torch.cuda.synchronize()
    assert abi.mxfp4_last_device_error() == abi.MXFP4_OK
    for out, ref in zip(outs, refs):
        assert torch.equal(out.view(torch.uint8).cpu(), ref.view(torch.uint8).cpu())


def oracle_hybrid_backward(t, rows_dx=None, rows_dw=None):
    """dX = dY . W and dW = dY^T . X through the oracle's tensorwise E5M2 and FP8 GEMM."""
    dyr, dyc, _, sdy = oracle.fp8_quantize_tw(workloads.bf16_bits(t["dY"]))
    _, xc, _, sx = oracle.fp8_quantize_tw(workloads.bf16_bits(t["X"]), row=False)
    _, wc, _, sw = oracle.fp8_quantize_tw(workloads.bf16_bits(t["W"]), row=False)
    M, N = t["dY"].shape
    dx = oracle.fp8_gemm(dyr, sdy, wc, sw, N, rows=rows_dx)
    dw = oracle.fp8_gemm(dyc, sdy, xc, sx, M, rows=rows_dw)
    return dx, dw


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_hybrid_backward_tiny(out_dtype):
    wl = workloads.TINY
    lin = wl.linears[0]
    t = wl.tensors(0)
    layer = MXFP4Linear(lin.M, lin.N, lin.K, train=True, out_dtype=out_dtype, backward="fp8")
    y, dx, dw = layer.step(t["X"].cuda(), t["W"].cuda(), t["dY"].cuda())
    torch.cuda.synchronize()
    assert abi.mxfp4_last_device_error() == abi.MXFP4_OK
    (cx, ax), (cw, aw) = oracle_hybrid_backward(t)
    check_gemm(dx, cx, ax, "hybrid dgrad")
    check_gemm(dw, cw, aw, "hybrid wgrad")
    # the forward is the MXFP4 one
    X, W = (oracle.quantize_row(workloads.bf16_bits(t[k])) for k in ("X", "W"))
    c, cabs = oracle.gemm(X[0], X[1], W[0], W[1])
    check_gemm(y, c, cabs, "hybrid fwd")


def test_hybrid_backward_flux_mlp_sampled():
    wl = workloads.FLUX_MLP_STEP
    lin = wl.linears[0]
    t = wl.tensors(0)
    layer = MXFP4Linear(lin.M, lin.N, lin.K, train=True, backward="fp8")
    _, dx, dw = layer.step(t["X"].cuda(), t["W"].cuda(), t["dY"].cuda())
    torch.cuda.synchronize()
    assert abi.mxfp4_last_device_error() == abi.MXFP4_OK
    rdx = np.array([0, 1, 127, 128, 2047, 4607])
    rdw = np.array([0, 255, 256, 6000, 12287])
    (cx, ax), (cw, aw) = oracle_hybrid_backward(t, rdx, rdw)
    check_gemm(dx[torch.as_tensor(rdx, device="cuda")], cx, ax, "flux hybrid dgrad")
    check_gemm(dw[torch.as_tensor(rdw, device="cuda")], cw, aw, "flux hybrid wgrad")


def test_fp8_quantize_batch_equals_single_calls():
    # One batched call over 1..3 tensors (row and/or column copies) gives each tensor its
    # own call's bytes and scalars.
    shapes = [((384, 1000), True, True), ((129, 200), False, True), ((640, 384), True, False)]
    xs = [pitched(workloads.student_t3(s, 0.1 * (i + 1), 801 + i)) for i, (s, _, _) in enumerate(shapes)]
    singles = []
    for x, (_, row, col) in zip(xs, shapes):
        qr, qc, amax, inv = abi.fp8_quantize(x, row=row, col=col)
        singles.append((qr, qc, amax.clone(), inv.clone()))
    torch.cuda.synchronize()
    for n in (1, 2, 3):
        tasks, outs = [], []
        sc = torch.full((2 * n,), float("nan"), dtype=torch.float32, device="cuda")
        for i, (x, (_, row, col)) in enumerate(zip(xs[:n], shapes[:n])):
            M, K = x.shape
            qr = torch.full((M, abi.fp8_pitch(K)), 0xAB, dtype=torch.uint8, device="cuda") if row else None
            qc = torch.full((K, abi.fp8_pitch(M)), 0xAB, dtype=torch.uint8, device="cuda") if col else None
            tasks.append((x, M, K, x.stride(0), qr, qc, sc[2 * i:2 * i + 1], sc[2 * i + 1:2 * i + 2]))
            outs.append((qr, qc, sc[2 * i:2 * i + 1], sc[2 * i + 1:2 * i + 2]))
        abi.mxfp4_fp8_quantize_tw_batch(tasks)
        torch.cuda.synchronize()
        assert abi.mxfp4_last_device_error() == abi.MXFP4_OK
        for got, want in zip(outs, singles[:n]):
            for g, w in zip(got, want):
                assert (g is None) == (w is None)
                if g is not None:
                    assert torch.equal(g.view(torch.uint8).cpu(), w.view(torch.uint8).cpu())


@pytest.mark.parametrize("bad", [float("inf"), float("-inf"), float("nan")])
def test_fp8_non_finite_input_is_reported(bad):
    # A non-finite element makes the tensor's amax non-finite: the conversion records it in
    # the device error word, which reads back as MXFP4_ERR_NONFINITE once and is then clear;
    # a finite tensor quantized afterwards is unaffected.
    x = workloads.normal((130, 200), 1.0, 5)
    x[77, 123] = bad
    abi.fp8_quantize(x.cuda())
    assert abi.mxfp4_last_device_error() == abi.MXFP4_ERR_NONFINITE
    assert abi.mxfp4_last_device_error() == abi.MXFP4_OK
    y = workloads.normal((130, 200), 1.0, 6)
    qr, qc, amax, inv = abi.fp8_quantize(y.cuda())
    assert abi.mxfp4_last_device_error() == abi.MXFP4_OK
    want_qr, want_qc, want_amax, want_inv = oracle.fp8_quantize_tw(workloads.bf16_bits(y))
    assert_bytes_equal(qr.cpu().numpy(), want_qr, "finite tensor after a non-finite one")


def test_quantize_batch_amax_output_feeds_the_fp8_quantizer():
    # The MXFP4 quantizer's tensor amax equals the FP8 quantizer's own amax pass (bit for
    # bit), and the FP8 quantization with amax_given gives the same codes and scale_inv.
    from mxfp4_block_scaled_quantize_gb300 import workloads
    for M, K, seed in ((300, 520, 1), (4608, 3072, 2), (77, 40, 3)):
        x = workloads.student_t3((M, K), 0.3, seed)
        ld = (K + 7) // 8 * 8
        xg = torch.zeros((M, ld), dtype=torch.bfloat16, device="cuda")
        xg[:, :K] = x.cuda()
        xg = xg[:, :K]
        rq, rs = abi.alloc_blob(M, K)
        amax = torch.full((1,), 123.0, dtype=torch.float32, device="cuda")   # zeroed by the call
        abi.mxfp4_quantize_batch([(xg, M, K, ld, rq, rs, None, None, 0, 0, amax)], False)
        p = abi.fp8_pitch
        qa = torch.empty((K, p(M)), dtype=torch.uint8, device="cuda")
        qb = torch.empty_like(qa)
        sa = torch.zeros(2, dtype=torch.float32, device="cuda")
        sb = torch.zeros(2, dtype=torch.float32, device="cuda")
        sb[0] = amax[0]
        abi.mxfp4_fp8_quantize_tw_batch([(xg, M, K, ld, None, qa, sa[0:1], sa[1:2])])
        abi.mxfp4_fp8_quantize_tw_batch([(xg, M, K, ld, None, qb, sb[0:1], sb[1:2], True)])
        torch.cuda.synchronize()
        assert abi.mxfp4_last_device_error() == abi.MXFP4_OK
        want = x.float().abs().max().item()
        assert amax.item() == want and sa[0].item() == want
        assert torch.equal(qa, qb) and torch.equal(sa, sb)
