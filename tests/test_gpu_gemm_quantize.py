"""GPU parity of the GEMM whose epilogue quantizes its own bf16 output (the next layer's
MXFP4 blobs): C against the fp64 oracle GEMM and bit-for-bit against the plain GEMM, and
the blobs byte for byte against the oracle's quantization of that same C (the integer
decisions are taken from C's bf16 values on both sides)."""
import numpy as np
import pytest
import torch

import oracle
from mxfp4_block_scaled_quantize_gb300 import abi, workloads
from parity import assert_bytes_equal, check_gemm, gather_tc_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield
    assert abi.mxfp4_last_device_error() == abi.MXFP4_OK


def _operands(M, N, K, seed):
    a = workloads.student_t3((M, K), 1.0, seed)
    b = workloads.normal((N, K), 0.05, seed + 1)
    ld = (K + 7) // 8 * 8
    ga = torch.zeros((M, ld), dtype=torch.bfloat16, device="cuda")
    gb = torch.zeros((N, ld), dtype=torch.bfloat16, device="cuda")
    ga[:, :K] = a.cuda()
    gb[:, :K] = b.cuda()
    aq, a_s = abi.quantize(ga[:, :K], dual=False)
    bq, b_s = abi.quantize(gb[:, :K], dual=False)
    return a, b, (aq, a_s, bq, b_s)


def _check_blobs_full(c_bits, outs, dual, what):
    rq, rs = oracle.quantize_row(c_bits)
    assert_bytes_equal(outs[0].cpu().numpy(), rq, f"{what} row q")
    assert_bytes_equal(outs[1].cpu().numpy().reshape(-1), oracle.scale_to_tc(rs).reshape(-1), f"{what} row s")
    if dual:
        cq, cs = oracle.quantize_col(c_bits)
        assert_bytes_equal(outs[2].cpu().numpy(), cq, f"{what} col q")
        assert_bytes_equal(outs[3].cpu().numpy().reshape(-1), oracle.scale_to_tc(cs).reshape(-1), f"{what} col s")


@pytest.mark.parametrize("M,N,K", [(300, 200, 264), (256, 256, 512), (129, 136, 128), (100, 72, 64),
                                   (520, 1000, 384), (4600, 384, 256), (1, 8, 32)])
@pytest.mark.parametrize("dual", [True, False])
@pytest.mark.parametrize("with_bias", [False, True])
def test_gemm_quantize_ragged(M, N, K, dual, with_bias):
    a, b, ops = _operands(M, N, K, M + 3 * N + K)
    ldc = (N + 7) // 8 * 8
    bias = workloads.normal((N,), 0.5, N).cuda() if with_bias else None
    c = torch.full((M, ldc), float("nan"), dtype=torch.bfloat16, device="cuda")
    # uninitialised-looking blob buffers: every byte must be written
    rq, rs = abi.alloc_blob(M, N)
    rq.fill_(0xA5)
    rs.fill_(0xA5)
    cq, cs = abi.alloc_blob(N, M) if dual else (None, None)
    if dual:
        cq.fill_(0x5A)
        cs.fill_(0x5A)
    abi.mxfp4_gemm_quantize(*ops, M, N, K, bias, c, ldc, rq, rs, cq, cs)
    # the plain GEMM (with its bias) into another buffer
    ref = torch.full((M, ldc), float("nan"), dtype=torch.bfloat16, device="cuda")
    if with_bias:
        abi.mxfp4_gemm_bias(*ops, M, N, K, bias, ref, ldc)
    else:
        abi.mxfp4_gemm(*ops, M, N, K, ref, ldc, abi.MXFP4_OUT_BF16)
    torch.cuda.synchronize()
    assert abi.mxfp4_last_device_error() == abi.MXFP4_OK
    what = f"gemm+quant {M}x{N}x{K} dual={dual} bias={with_bias}"
    assert torch.equal(c[:, :N].view(torch.int16), ref[:, :N].view(torch.int16)), what
    if not with_bias:
        ab, bb = workloads.bf16_bits(a), workloads.bf16_bits(b)
        want, wabs = oracle.gemm(*oracle.quantize_row(ab), *oracle.quantize_row(bb))
        check_gemm(c[:, :N], want, wabs, what)
    c_bits = workloads.bf16_bits(c[:, :N].cpu())
    _check_blobs_full(c_bits, (rq, rs, cq, cs), dual, what)


def test_gemm_quantize_equals_quantizer_on_its_output():
    # The same bytes as the library's own dual quantizer run on the GEMM's output.
    M, N, K = 700, 640, 512
    _, _, ops = _operands(M, N, K, 9)
    c, rq, rs, cq, cs = abi.gemm_quantize(*ops, M, N, K, dual=True)
    want = abi.quantize(c, dual=True)
    torch.cuda.synchronize()
    for got, exp in zip((rq, rs, cq, cs), want):
        assert torch.equal(got, exp)


def test_gemm_quantize_flux_linear1_sampled():
    # The single-stream block's linear1 forward, 4608 x 21504 x 3072, with its output's
    # blobs: C bit-identical to the plain GEMM, sampled rows and columns of the blobs against
    # the oracle's quantization of those rows and columns of C.
    t = workloads.FLUX_SINGLE_BLOCK.tensors(0)
    M, K = t["X"].shape
    N = t["W"].shape[0]
    aq, a_s = abi.quantize(t["X"].cuda(), dual=False)
    bq, b_s = abi.quantize(t["W"].cuda(), dual=False)
    c, rq, rs, cq, cs = abi.gemm_quantize(aq, a_s, bq, b_s, M, N, K, dual=True)
    ref = abi.gemm(aq, a_s, bq, b_s, M, N, K)
    torch.cuda.synchronize()
    assert abi.mxfp4_last_device_error() == abi.MXFP4_OK
    assert torch.equal(c.view(torch.int16), ref.view(torch.int16))
    cb = workloads.bf16_bits(c.cpu())
    rng = np.random.default_rng(21)
    rows = np.unique(np.concatenate([rng.choice(M, 12, replace=False), [0, M - 1]]))
    cols = np.unique(np.concatenate([rng.choice(N, 12, replace=False), [0, N - 1]]))
    q, s = oracle.quantize_row(np.ascontiguousarray(cb[rows]))
    assert_bytes_equal(rq[torch.as_tensor(rows, device="cuda")].cpu().numpy(), q, "flux out row q")
    assert_bytes_equal(gather_tc_rows(rs.cpu().numpy(), rows, s.shape[1]), s, "flux out row s")
    q, s = oracle.quantize_col(np.ascontiguousarray(cb[:, cols]))
    assert_bytes_equal(cq[torch.as_tensor(cols, device="cuda")].cpu().numpy(), q, "flux out col q")
    assert_bytes_equal(gather_tc_rows(cs.cpu().numpy(), cols, s.shape[1]), s, "flux out col s")

