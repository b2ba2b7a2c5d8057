"""GPU parity of the quantizer with the QK RMSNorm + interleaved RoPE backward in its staging
read: the bf16 d(mixed_qkv) it computes against the fp64 oracle (within the fp32 bound), and
its blobs byte for byte against the oracle's quantization of that same bf16 d(mixed_qkv)."""
import numpy as np
import pytest
import torch

import oracle
from mxfp4_block_scaled_quantize_gb300 import abi, workloads
from parity import assert_bytes_equal, gather_tc_rows

pytestmark = pytest.mark.gpu
D = 128


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield
    assert abi.mxfp4_last_device_error() == abi.MXFP4_OK


def _case(M, H, seed):
    """mixed_qkv x ~ N(0, 1) (a GEMM output), its gradient g ~ N(0, 1e-3) with a few larger
    tokens, the forward's r from the oracle's forward, norm weights around 1, RoPE angles."""
    rng = np.random.default_rng(seed)
    x = workloads.normal((M, 3 * H * D), 1.0, seed)
    g = workloads.normal((M, 3 * H * D), 1e-3, seed + 1)
    xb, gb = workloads.bf16_bits(x), workloads.bf16_bits(g)
    wq = rng.uniform(0.5, 1.5, D).astype(np.float32)
    wk = rng.uniform(0.5, 1.5, D).astype(np.float32)
    theta = rng.uniform(-np.pi, np.pi, (M, D // 2))
    cs, sn = np.cos(theta).astype(np.float32), np.sin(theta).astype(np.float32)
    xv = (xb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    _, r = oracle.qk_norm_rope_fwd(xv, wq, wk, cs, sn, H, D)
    return x, g, xb, gb, r.astype(np.float32), wq, wk, cs, sn


def _run(x, g, r, wq, wk, cs, sn, H, layout=abi.MXFP4_SCALE_TC):
    dev = [torch.as_tensor(a).cuda() for a in (r, wq, wk, cs, sn)]
    outs = abi.quantize_qk_norm_rope_bwd(g.cuda(), x.cuda(), *dev, H, layout=layout, with_dmixed=True)
    torch.cuda.synchronize()
    assert abi.mxfp4_last_device_error() == abi.MXFP4_OK
    return outs


def _check_dmixed(dm_bits, want, what):
    """bf16 d(mixed_qkv) within one bf16 ulp of the exact value plus 2^-17 of the largest
    magnitude of its (token, head, part) row: fp32 evaluation with a 128-term dot product."""
    got = (dm_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    M, K = want.shape
    rowmax = np.abs(want).reshape(M, K // D, D).max(axis=2).repeat(D, axis=1)
    ulp = np.ldexp(1.0, np.floor(np.log2(np.maximum(np.abs(want), 1e-300))).astype(np.int64) - 7)
    bad = np.abs(got - want) > ulp + rowmax * 2.0 ** -17
    assert not bad.any(), f"{what}: {bad.sum()} elements outside the bound, first {np.argwhere(bad)[0]}"


@pytest.mark.parametrize("M,H", [(1, 1), (130, 1), (257, 2), (640, 3)])
@pytest.mark.parametrize("layout", [abi.MXFP4_SCALE_PLAIN, abi.MXFP4_SCALE_TC])
def test_norm_rope_prologue_small(M, H, layout):
    x, g, xb, gb, r, wq, wk, cs, sn = _case(M, H, 11 * M + H)
    rq, rs, cq, cs_, dm = _run(x, g, r, wq, wk, cs, sn, H, layout)
    want = oracle.qk_norm_rope_bwd(gb, xb, r, wq, wk, cs, sn, H, D)
    dmb = dm.cpu().view(torch.int16).numpy().view(np.uint16)
    _check_dmixed(dmb, want, f"dmixed {M}x{H}")
    for h in range(H):   # v is the gradient itself
        v = slice(h * 3 * D + 2 * D, h * 3 * D + 3 * D)
        assert np.array_equal(dmb[:, v], gb[:, v])
    tc = layout == abi.MXFP4_SCALE_TC
    q, s = oracle.quantize_row(dmb)
    assert_bytes_equal(rq.cpu().numpy(), q, "row q")
    assert_bytes_equal(rs.cpu().numpy().reshape(-1), (oracle.scale_to_tc(s) if tc else s).reshape(-1), "row s")
    q, s = oracle.quantize_col(dmb)
    assert_bytes_equal(cq.cpu().numpy(), q, "col q")
    assert_bytes_equal(cs_.cpu().numpy().reshape(-1), (oracle.scale_to_tc(s) if tc else s).reshape(-1), "col s")


def test_norm_rope_prologue_without_dmixed_gives_the_same_blobs():
    M, H = 300, 2
    x, g, xb, gb, r, wq, wk, cs, sn = _case(M, H, 5)
    a = _run(x, g, r, wq, wk, cs, sn, H)
    dev = [torch.as_tensor(t).cuda() for t in (r, wq, wk, cs, sn)]
    b = abi.quantize_qk_norm_rope_bwd(g.cuda(), x.cuda(), *dev, H)
    # and the plain dual quantizer over the written d(mixed_qkv) gives the same bytes again
    c = abi.quantize(a[4], dual=True)
    torch.cuda.synchronize()
    for u, v, w in zip(a[:4], b, c):
        assert torch.equal(u, v) and torch.equal(u, w)


def test_norm_rope_prologue_flux_qkv_sampled():
    # The Flux-12B QKV projection's gradient: M 4608 tokens, 24 heads (d(mixed_qkv)
    # [4608, 9216]), sampled rows and whole columns against the oracle.
    M, H = 4608, 24
    x, g, xb, gb, r, wq, wk, cs, sn = _case(M, H, 2024)
    rq, rs, cq, cs_, dm = _run(x, g, r, wq, wk, cs, sn, H)
    dmb = dm.cpu().view(torch.int16).numpy().view(np.uint16)
    rng = np.random.default_rng(3)
    rows = np.unique(np.concatenate([rng.choice(M, 16, replace=False), [0, M - 1]]))
    want = oracle.qk_norm_rope_bwd(np.ascontiguousarray(gb[rows]), np.ascontiguousarray(xb[rows]),
                                   np.ascontiguousarray(r[rows]), wq, wk, np.ascontiguousarray(cs[rows]),
                                   np.ascontiguousarray(sn[rows]), H, D)
    _check_dmixed(dmb[rows], want, "flux dmixed rows")
    q, s = oracle.quantize_row(np.ascontiguousarray(dmb[rows]))
    assert_bytes_equal(rq[torch.as_tensor(rows, device="cuda")].cpu().numpy(), q, "flux row q")
    assert_bytes_equal(gather_tc_rows(rs.cpu().numpy(), rows, s.shape[1]), s, "flux row s")
    cols = np.unique(np.concatenate([rng.choice(3 * H * D, 16, replace=False), [0, 3 * H * D - 1]]))
    q, s = oracle.quantize_col(np.ascontiguousarray(dmb[:, cols]))
    assert_bytes_equal(cq[torch.as_tensor(cols, device="cuda")].cpu().numpy(), q, "flux col q")
    assert_bytes_equal(gather_tc_rows(cs_.cpu().numpy(), cols, s.shape[1]), s, "flux col s")
