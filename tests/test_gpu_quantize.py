"""GPU parity of the MXFP4 quantizers (row-only and dual) against the CPU oracle.

Every comparison is byte-for-byte, padding and both scale layouts included.  The inputs
come from the seeded generators in mxfp4_block_scaled_quantize_gb300.workloads.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from mxfp4_block_scaled_quantize_gb300 import abi, workloads
from parity import (assert_bytes_equal, check_quantized_full, check_quantized_sampled,
                    check_rows_cols)

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
LAYOUTS = [abi.MXFP4_SCALE_PLAIN, abi.MXFP4_SCALE_TC]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield
    assert abi.mxfp4_last_device_error() == abi.MXFP4_OK


def quant(x_cpu, dual, layout, ldx=None):
    """Quantize a CPU bf16 tensor on the GPU (optionally from a wider row pitch)."""
    M, K = x_cpu.shape
    if ldx is not None and ldx != K:
        wide = torch.zeros((M, ldx), dtype=torch.bfloat16)
        wide[:, :K] = x_cpu
        xg = wide.cuda()[:, :K]
    else:
        xg = x_cpu.cuda()
    outs = abi.quantize(xg, dual=dual, layout=layout)
    torch.cuda.synchronize()
    assert abi.mxfp4_last_device_error() == abi.MXFP4_OK
    return outs


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("name", ["X", "W", "dY"])
def test_tiny_config_dual(name, layout):
    t = workloads.TINY.tensors(0)[name]
    check_quantized_full(t, quant(t, True, layout), layout, True, f"tiny {name}")


@pytest.mark.parametrize("layout", LAYOUTS)
def test_tiny_config_row_only(layout):
    t = workloads.TINY.tensors(0)["X"]
    check_quantized_full(t, quant(t, False, layout), layout, False, "tiny X row-only")


def _bits_to_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(bits.astype(np.uint16).view(np.int16)).view(torch.bfloat16)


def test_worked_examples():
    with open(os.path.join(GOLDEN, "mx_worked_examples.json")) as f:
        cases = json.load(f)["cases"]
    rows = []
    for case in cases:
        vals = np.zeros(32, np.float32)
        vals[:len(case["values"])] = case["values"]
        rows.append((vals.view(np.uint32) >> 16).astype(np.uint16))
    bits = np.stack(rows)                                  # one block per row
    x = _bits_to_bf16(bits)
    for layout in LAYOUTS:
        outs = quant(x, True, layout)
        check_quantized_full(x, outs, layout, True, "worked examples")
        rq = outs[0].cpu().numpy()
        rs = outs[1].cpu().numpy()
        for i, case in enumerate(cases):
            s = rs[i, 0] if layout == abi.MXFP4_SCALE_PLAIN else rs[(i % 32) * 16 + (i // 32) * 4]
            assert s == case["scale"], case["name"]
            codes = np.empty(32, np.uint8)
            codes[0::2] = rq[i, :16] & 0xF
            codes[1::2] = rq[i, :16] >> 4
            assert list(codes[:len(case["codes"])]) == case["codes"], case["name"]


@pytest.mark.parametrize("transpose", [False, True])
def test_every_finite_bf16_pattern(transpose):
    b = np.arange(0x10000, dtype=np.uint32).astype(np.uint16)
    finite = (b & 0x7F80) != 0x7F80
    b = np.where(finite, b, 0).astype(np.uint16)
    # mix magnitudes inside blocks: permute with a fixed seed so blocks span many binades
    rng = np.random.default_rng(7)
    b = b[rng.permutation(b.size)].reshape(2048, 32)
    if transpose:
        b = np.ascontiguousarray(b.T)
    x = _bits_to_bf16(b)
    for layout in LAYOUTS:
        check_quantized_full(x, quant(x, True, layout), layout, True, "all bf16 patterns")


def _edge_input(M, K, seed):
    x = workloads.student_t3((M, K), 1.0, seed)
    return workloads.inject_edge_blocks(x, seed + 1)


@pytest.mark.parametrize("M,K,ldx", [(1, 8, 8), (1, 32, 32), (32, 8, 16), (100, 40, 40),
                                     (130, 200, 200), (257, 33, 40), (256, 512, 520),
                                     (128, 128, 128), (129, 129, 136), (640, 384, 384),
                                     (4600, 256, 256)])
def test_ragged_shapes(M, K, ldx):
    x = _edge_input(M, K, M * 7 + K)
    for layout in LAYOUTS:
        check_quantized_full(x, quant(x, True, layout, ldx), layout, True, f"dual {M}x{K}")
        check_quantized_full(x, quant(x, False, layout, ldx), layout, False, f"row {M}x{K}")


@pytest.mark.parametrize("dual", [True, False])
@pytest.mark.parametrize("layout", LAYOUTS)
def test_batch_equals_single_calls(dual, layout):
    # One launch over 1..4 tensors of different shapes (ragged edges, a pitched input) gives
    # each tensor the bytes its own call gives.
    shapes = [(300, 200, 200), (129, 1000, 1008), (1, 40, 40), (640, 384, 392)]
    xs = [_edge_input(M, K, 31 * i + M) for i, (M, K, _) in enumerate(shapes)]
    singles = [quant(x, dual, layout, ldx) for x, (_, _, ldx) in zip(xs, shapes)]
    for n in (1, 2, 4):
        tasks, outs = [], []
        for x, (M, K, ldx) in zip(xs[:n], shapes[:n]):
            wide = torch.zeros((M, ldx), dtype=torch.bfloat16)
            wide[:, :K] = x
            xg = wide.cuda()
            rq, rs = abi.alloc_blob(M, K, layout)
            cq, cs = abi.alloc_blob(K, M, layout) if dual else (None, None)
            tasks.append((xg, M, K, ldx, rq, rs, cq, cs))
            outs.append((rq, rs, cq, cs) if dual else (rq, rs))
        abi.mxfp4_quantize_batch(tasks, dual, layout)
        torch.cuda.synchronize()
        assert abi.mxfp4_last_device_error() == abi.MXFP4_OK
        for got, want in zip(outs, singles):
            for g, w in zip(got, want):
                assert torch.equal(g.cpu(), w.cpu())


def test_row_only_equals_row_half_of_dual():
    x = _edge_input(4608, 3072, 11)
    r = quant(x, False, abi.MXFP4_SCALE_TC)
    d = quant(x, True, abi.MXFP4_SCALE_TC)
    assert torch.equal(r[0], d[0]) and torch.equal(r[1], d[1])


def test_outputs_written_exactly():
    """Guard bytes around every output stay untouched; padding is written (buffers start
    as 0xA5 garbage)."""
    M, K = 300, 200
    x = _edge_input(M, K, 5).cuda()
    guard = 4096
    for layout in LAYOUTS:
        sizes = [abi.mxfp4_quantize_sizes(M, K, layout), abi.mxfp4_quantize_sizes(K, M, layout)]
        bufs = []
        for qb, sb in sizes:
            for nb in (qb, sb):
                t = torch.full((nb + 2 * guard,), 0xA5, dtype=torch.uint8, device="cuda")
                bufs.append(t)
        views = [b[guard:-guard] for b in bufs]
        abi.mxfp4_quantize_dual(x, M, K, K, views[0], views[1], views[2], views[3], layout)
        torch.cuda.synchronize()
        for b in bufs:
            assert torch.all(b[:guard] == 0xA5) and torch.all(b[-guard:] == 0xA5)
        Kp, Mp = oracle.padded(K), oracle.padded(M)
        outs = [views[0].view(M, Kp // 2), views[1], views[2].view(K, Mp // 2), views[3]]
        if layout == abi.MXFP4_SCALE_PLAIN:
            outs[1] = outs[1].view(M, Kp // 32)
            outs[3] = outs[3].view(K, Mp // 32)
        check_quantized_full(x.cpu(), outs, layout, True, f"guarded layout {layout}")


@pytest.mark.parametrize("M", workloads.SWEEP_M)
@pytest.mark.parametrize("K", workloads.SWEEP_K)
@pytest.mark.parametrize("scale", workloads.SWEEP_SCALE)
def test_sweep_sampled(M, K, scale):
    # The whole bandwidth/edge sweep: every M x K pair at every scale, Student-t(3) values
    # with all-subnormal, mixed, near-bf16-max and all-zero blocks along both packings, in
    # the launch configuration of the full-size call; sampled rows and whole columns.
    x = workloads.sweep_tensor(M, K, scale)
    outs = quant(x, True, abi.MXFP4_SCALE_TC)
    n = 16 if M * K > 10**8 else 48
    check_quantized_sampled(x, outs, True, f"sweep {M}x{K}x{scale}", n_rows=n, n_cols=n)
    # the injected edge blocks sit in rows 7 + 13i and columns 11 + 17i: always compared
    edge_rows = np.array([(7 + 13 * i) % M for i in range(4)])
    edge_cols = np.array([(11 + 17 * i) % K for i in range(4)])
    check_rows_cols(x, outs, edge_rows, edge_cols, f"sweep {M}x{K}x{scale} edge blocks")


@pytest.mark.parametrize("wname", ["flux12b_qkv_fwd_4608x9216x3072",
                                   "flux12b_mlp_up_train_step_4608x12288x3072"])
def test_flux_tensors_sampled(wname):
    wl = workloads.WORKLOADS[wname]
    t = wl.tensors(0)
    dual = wl.linears[0].train
    for name, x in t.items():
        check_quantized_sampled(x, quant(x, dual, abi.MXFP4_SCALE_TC), dual, f"{wname} {name}")


def test_argument_errors():
    x = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    q, s = abi.alloc_blob(64, 64)
    lib = abi.load()
    st = lib.mxfp4_quantize(x.data_ptr() + 2, 64, 64, 64, q.data_ptr(), s.data_ptr(), 1, None)
    assert st == abi.MXFP4_ERR_MISALIGNED
    st = lib.mxfp4_quantize(x.data_ptr(), 64, 60, 60, q.data_ptr(), s.data_ptr(), 1, None)
    assert st == abi.MXFP4_ERR_MISALIGNED          # row pitch not a multiple of 8
    st = lib.mxfp4_quantize(x.data_ptr(), 64, 64, 32, q.data_ptr(), s.data_ptr(), 1, None)
    assert st == abi.MXFP4_ERR_INVALID_ARG         # ldx < K
    st = lib.mxfp4_quantize(x.data_ptr(), 0, 64, 64, q.data_ptr(), s.data_ptr(), 1, None)
    assert st == abi.MXFP4_ERR_INVALID_ARG
    st = lib.mxfp4_quantize(x.data_ptr(), 64, 64, 64, q.data_ptr(), s.data_ptr(), 7, None)
    assert st == abi.MXFP4_ERR_INVALID_ARG


def test_bounded_wait_reports_timeout_and_context_survives():
    abi.mxfp4_selftest_bounded_wait(20_000_000)     # 20 ms
    assert abi.mxfp4_last_device_error() == abi.MXFP4_ERR_TIMEOUT
    assert abi.mxfp4_last_device_error() == abi.MXFP4_OK   # the word was cleared
    t = workloads.TINY.tensors(0)["X"]
    check_quantized_full(t, quant(t, True, abi.MXFP4_SCALE_TC), abi.MXFP4_SCALE_TC, True,
                         "after timeout")


# --- stochastic rounding (the gradient quantizer's `use_sr`) ----------------------------

def quant_sr(x_cpu, layout, seed, ldx=None):
    M, K = x_cpu.shape
    if ldx is not None and ldx != K:
        wide = torch.zeros((M, ldx), dtype=torch.bfloat16)
        wide[:, :K] = x_cpu
        xg = wide.cuda()[:, :K]
    else:
        xg = x_cpu.cuda()
    outs = abi.quantize(xg, dual=True, layout=layout, sr_seed=seed)
    torch.cuda.synchronize()
    assert abi.mxfp4_last_device_error() == abi.MXFP4_OK
    return outs


def check_sr_full(x_cpu, outs, layout, seed, what):
    xb = workloads.bf16_bits(x_cpu)
    rq, rs, cq, cs = oracle.quantize_dual_sr(xb, seed)
    tc = layout == abi.MXFP4_SCALE_TC
    assert_bytes_equal(outs[0].cpu().numpy(), rq, f"{what} row q")
    assert_bytes_equal(outs[1].cpu().numpy().reshape(-1), (oracle.scale_to_tc(rs) if tc else rs).reshape(-1),
                       f"{what} row s")
    assert_bytes_equal(outs[2].cpu().numpy(), cq, f"{what} col q")
    assert_bytes_equal(outs[3].cpu().numpy().reshape(-1), (oracle.scale_to_tc(cs) if tc else cs).reshape(-1),
                       f"{what} col s")


@pytest.mark.parametrize("M,K,ldx", [(1, 8, 8), (32, 8, 16), (100, 40, 40), (130, 200, 200),
                                     (257, 33, 40), (256, 512, 520), (129, 129, 136), (640, 384, 384)])
@pytest.mark.parametrize("seed", [0, 0x9E3779B97F4A7C15])
def test_sr_ragged_shapes(M, K, ldx, seed):
    # Every byte of both blobs equals the oracle's stochastic rounding with the same seed
    # (Philox bits, threshold rule and counter layout), edge blocks included.
    x = _edge_input(M, K, 3 * M + K)
    for layout in LAYOUTS:
        check_sr_full(x, quant_sr(x, layout, seed, ldx), layout, seed, f"sr {M}x{K} seed {seed:#x}")


def test_sr_every_finite_bf16_pattern():
    b = np.arange(0x10000, dtype=np.uint32).astype(np.uint16)
    fin = (b & 0x7F80) != 0x7F80
    b = b[fin]
    n = (b.size + 255) // 256 * 256
    pad = np.zeros(n, np.uint16)
    pad[:b.size] = b
    x = _bits_to_bf16(pad.reshape(-1, 256))   # rows of 256: a 16-byte row pitch
    check_sr_full(x, quant_sr(x, abi.MXFP4_SCALE_TC, 12345), abi.MXFP4_SCALE_TC, 12345, "sr all bf16")


def test_sr_seed_behaviour():
    # Same seed: identical bytes; another seed: different elements, the same scales.
    x = workloads.normal((384, 640), 1.0, 77).cuda()
    a = abi.quantize(x, dual=True, sr_seed=5)
    b = abi.quantize(x, dual=True, sr_seed=5)
    c = abi.quantize(x, dual=True, sr_seed=6)
    n = abi.quantize(x, dual=True)
    torch.cuda.synchronize()
    for u, v in zip(a, b):
        assert torch.equal(u, v)
    assert not torch.equal(a[0], c[0]) and not torch.equal(a[2], c[2])
    assert torch.equal(a[1], n[1]) and torch.equal(a[3], n[3])


def test_sr_flux_dy_sampled():
    # The Flux-12B MLP gradient dY [4608, 12288] in the launch configuration of the
    # backward step, against the oracle on sampled rows and columns at their true positions.
    wl = workloads.FLUX_MLP_STEP
    dy = wl.tensors(0)["dY"]
    seed = 2026
    outs = quant_sr(dy, abi.MXFP4_SCALE_TC, seed)
    xb = workloads.bf16_bits(dy)
    M, K = xb.shape
    rng = np.random.default_rng(3)
    rows = np.unique(np.concatenate([rng.choice(M, 24, replace=False), [0, 127, 128, M - 1]]))
    cols = np.unique(np.concatenate([rng.choice(K, 24, replace=False), [0, 1, K - 2, K - 1]]))
    rq, rs = oracle.quantize_row_sr(np.ascontiguousarray(xb[rows]), seed, row_ids=rows)
    assert_bytes_equal(outs[0][torch.as_tensor(rows, device="cuda")].cpu().numpy(), rq, "sr dY row q")
    from parity import gather_tc_rows
    assert_bytes_equal(gather_tc_rows(outs[1].cpu().numpy(), rows, rs.shape[1]), rs, "sr dY row s")
    cq, cs = oracle.quantize_col_sr(np.ascontiguousarray(xb[:, cols]), seed, col_ids=cols)
    assert_bytes_equal(outs[2][torch.as_tensor(cols, device="cuda")].cpu().numpy(), cq, "sr dY col q")
    assert_bytes_equal(gather_tc_rows(outs[3].cpu().numpy(), cols, cs.shape[1]), cs, "sr dY col s")


# --- 2-D (32 x 32) block scales (the weight recipe of `_quantize_weight_dual`) -----------

def check_2d_full(x_cpu, outs, layout, dual, what):
    xb = workloads.bf16_bits(x_cpu)
    rq, rs = oracle.quantize_row_2d(xb)
    tc = layout == abi.MXFP4_SCALE_TC
    assert_bytes_equal(outs[0].cpu().numpy(), rq, f"{what} row q")
    assert_bytes_equal(outs[1].cpu().numpy().reshape(-1), (oracle.scale_to_tc(rs) if tc else rs).reshape(-1),
                       f"{what} row s")
    if dual:
        cq, cs = oracle.quantize_col_2d(xb)
        assert_bytes_equal(outs[2].cpu().numpy(), cq, f"{what} col q")
        assert_bytes_equal(outs[3].cpu().numpy().reshape(-1), (oracle.scale_to_tc(cs) if tc else cs).reshape(-1),
                           f"{what} col s")


def quant_2d(x_cpu, dual, layout, ldx=None):
    M, K = x_cpu.shape
    if ldx is not None and ldx != K:
        wide = torch.zeros((M, ldx), dtype=torch.bfloat16)
        wide[:, :K] = x_cpu
        xg = wide.cuda()[:, :K]
    else:
        xg = x_cpu.cuda()
    outs = abi.quantize(xg, dual=dual, layout=layout, block_2d=True)
    torch.cuda.synchronize()
    assert abi.mxfp4_last_device_error() == abi.MXFP4_OK
    return outs


@pytest.mark.parametrize("M,K,ldx", [(1, 8, 8), (32, 32, 32), (33, 40, 40), (100, 40, 40), (130, 200, 200),
                                     (257, 33, 40), (256, 512, 520), (129, 129, 136), (640, 384, 384),
                                     (4600, 256, 256)])
def test_2d_blocks_ragged_shapes(M, K, ldx):
    # Every byte of both blobs (and of the row-only blob) equals the oracle's 2-D block
    # quantization, edge blocks and ragged 32 x 32 blocks at the right and bottom included.
    x = _edge_input(M, K, 5 * M + K)
    for layout in LAYOUTS:
        check_2d_full(x, quant_2d(x, True, layout, ldx), layout, True, f"2d dual {M}x{K}")
        check_2d_full(x, quant_2d(x, False, layout, ldx), layout, False, f"2d row {M}x{K}")


def test_2d_blocks_every_finite_bf16_pattern():
    b = np.arange(0x10000, dtype=np.uint32).astype(np.uint16)
    b = np.where((b & 0x7F80) != 0x7F80, b, 0).astype(np.uint16)
    rng = np.random.default_rng(9)
    b = b[rng.permutation(b.size)].reshape(256, 256)
    x = _bits_to_bf16(b)
    for layout in LAYOUTS:
        check_2d_full(x, quant_2d(x, True, layout), layout, True, "2d all bf16 patterns")


def test_2d_blocks_mixed_batch_equals_single_calls():
    # X with 1 x 32 blocks and W with 32 x 32 blocks in one launch (the layer's forward
    # quantization with the weight recipe) give the bytes of their own calls.
    x = _edge_input(300, 200, 41)
    w = _edge_input(520, 200, 43)
    sx = quant(x, True, abi.MXFP4_SCALE_TC)
    sw = quant_2d(w, True, abi.MXFP4_SCALE_TC)
    bx = [abi.alloc_blob(300, 200), abi.alloc_blob(200, 300)]
    bw = [abi.alloc_blob(520, 200), abi.alloc_blob(200, 520)]
    xg, wg = x.cuda(), w.cuda()
    abi.mxfp4_quantize_batch([(xg, 300, 200, 200, *bx[0], *bx[1], 0),
                              (wg, 520, 200, 200, *bw[0], *bw[1], abi.MXFP4_QUANT_2D_BLOCKS)], True)
    torch.cuda.synchronize()
    assert abi.mxfp4_last_device_error() == abi.MXFP4_OK
    for got, want in zip([*bx[0], *bx[1]], sx):
        assert torch.equal(got.cpu(), want.cpu())
    for got, want in zip([*bw[0], *bw[1]], sw):
        assert torch.equal(got.cpu(), want.cpu())


@pytest.mark.parametrize("li", [0, 1])
def test_2d_blocks_flux_weights_sampled(li):
    # The single-stream block's weights W1 [21504, 3072] and W2 [3072, 15360]: whole 32-row
    # bands (row blob) and 32-column bands (col blob) quantized by the oracle at their true
    # positions.
    w = workloads.FLUX_SINGLE_BLOCK.tensors(li)["W"]
    outs = quant_2d(w, True, abi.MXFP4_SCALE_TC)
    wb = workloads.bf16_bits(w)
    N, K = wb.shape
    from parity import gather_tc_rows
    for band in (0, (N // 32) // 2, N // 32 - 1):
        rows = np.arange(32 * band, min(N, 32 * band + 32))
        rq, rs = oracle.quantize_row_2d(np.ascontiguousarray(wb[rows]))
        assert_bytes_equal(outs[0][torch.as_tensor(rows, device="cuda")].cpu().numpy(), rq, f"W{li + 1} 2d row q")
        assert_bytes_equal(gather_tc_rows(outs[1].cpu().numpy(), rows, rs.shape[1]), rs, f"W{li + 1} 2d row s")
    for band in (0, (K // 32) // 2, K // 32 - 1):
        cols = np.arange(32 * band, min(K, 32 * band + 32))
        cq, cs = oracle.quantize_col_2d(np.ascontiguousarray(wb[:, cols]))
        assert_bytes_equal(outs[2][torch.as_tensor(cols, device="cuda")].cpu().numpy(), cq, f"W{li + 1} 2d col q")
        assert_bytes_equal(gather_tc_rows(outs[3].cpu().numpy(), cols, cs.shape[1]), cs, f"W{li + 1} 2d col s")


# --- Hadamard transform of the column blob (`colwise_use_rht`) ---------------------------

RHT_MASKS = (0x0000, 0xA5C3, 0xFFFF, 0x8001)


def _rht_input(M, K, seed):
    """Student-t values with subnormal, mixed and zero blocks (edge kinds), magnitudes kept
    below 2^100 so that no 16-row sum can overflow."""
    x = _edge_input(M, K, seed).float()
    x = torch.where(x.abs() > 2.0 ** 100, x * 2.0 ** -120, x)
    return x.to(torch.bfloat16)


def check_rht_full(x_cpu, outs, layout, signs, what):
    xb = workloads.bf16_bits(x_cpu)
    tc = layout == abi.MXFP4_SCALE_TC
    rq, rs = oracle.quantize_row(xb)
    assert_bytes_equal(outs[0].cpu().numpy(), rq, f"{what} row q")
    assert_bytes_equal(outs[1].cpu().numpy().reshape(-1), (oracle.scale_to_tc(rs) if tc else rs).reshape(-1),
                       f"{what} row s")
    cq, cs = oracle.quantize_col_rht(xb, signs)
    assert_bytes_equal(outs[2].cpu().numpy(), cq, f"{what} col q")
    assert_bytes_equal(outs[3].cpu().numpy().reshape(-1), (oracle.scale_to_tc(cs) if tc else cs).reshape(-1),
                       f"{what} col s")


@pytest.mark.parametrize("M,K,ldx", [(1, 8, 8), (16, 32, 32), (40, 40, 40), (100, 40, 40), (130, 200, 200),
                                     (257, 33, 40), (256, 512, 520), (640, 384, 384), (4600, 256, 256)])
@pytest.mark.parametrize("signs", RHT_MASKS)
def test_rht_ragged_shapes(M, K, ldx, signs):
    # Row blob as the plain dual quantizer, col blob as the oracle's transformed columns,
    # byte for byte (groups straddling M included).
    x = _rht_input(M, K, 3 * M + 5 * K)
    for layout in LAYOUTS:
        wide = torch.zeros((M, ldx), dtype=torch.bfloat16)
        wide[:, :K] = x
        outs = abi.quantize(wide.cuda()[:, :K], dual=True, layout=layout, rht_signs=signs)
        torch.cuda.synchronize()
        assert abi.mxfp4_last_device_error() == abi.MXFP4_OK
        check_rht_full(x, outs, layout, signs, f"rht {M}x{K} signs {signs:#06x}")


def test_rht_every_bf16_pattern_below_overflow():
    b = np.arange(0x10000, dtype=np.uint32).astype(np.uint16)
    b = np.where((b & 0x7F80) < (200 << 7), b, 0).astype(np.uint16)    # exponent field < 200
    rng = np.random.default_rng(13)
    x = _bits_to_bf16(b[rng.permutation(b.size)].reshape(256, 256))
    for signs in RHT_MASKS:
        outs = abi.quantize(x.cuda(), dual=True, layout=abi.MXFP4_SCALE_TC, rht_signs=signs)
        torch.cuda.synchronize()
        check_rht_full(x, outs, abi.MXFP4_SCALE_TC, signs, f"rht all patterns {signs:#06x}")


def test_rht_flux_activation_sampled():
    # Flux X [4608, 3072] and the GELU-like H [4608, 15360]: whole sampled columns of the col
    # blob against the oracle's transform of those columns.
    from parity import gather_tc_rows
    for li in (0, 1):
        x = workloads.FLUX_SINGLE_BLOCK.tensors(li)["X"]
        outs = abi.quantize(x.cuda(), dual=True, layout=abi.MXFP4_SCALE_TC, rht_signs=0xA5C3)
        torch.cuda.synchronize()
        xb = workloads.bf16_bits(x)
        K = xb.shape[1]
        cols = np.unique(np.concatenate([np.random.default_rng(li).choice(K, 24, replace=False), [0, K - 1]]))
        cq, cs = oracle.quantize_col_rht(np.ascontiguousarray(xb[:, cols]), 0xA5C3)
        assert_bytes_equal(outs[2][torch.as_tensor(cols, device="cuda")].cpu().numpy(), cq, f"flux {li} rht col q")
        assert_bytes_equal(gather_tc_rows(outs[3].cpu().numpy(), cols, cs.shape[1]), cs, f"flux {li} rht col s")


def test_recipes_mixed_batch_equals_single_calls():
    # The layer's forward quantization with both recipes: X with the transformed col blob and
    # W with 2-D blocks in one launch give the bytes of their own calls.
    x = _rht_input(300, 200, 51)
    w = _edge_input(520, 200, 53)
    sx = abi.quantize(x.cuda(), dual=True, rht_signs=0x1357)
    sw = quant_2d(w, True, abi.MXFP4_SCALE_TC)
    bx = [abi.alloc_blob(300, 200), abi.alloc_blob(200, 300)]
    bw = [abi.alloc_blob(520, 200), abi.alloc_blob(200, 520)]
    abi.mxfp4_quantize_batch([(x.cuda(), 300, 200, 200, *bx[0], *bx[1], abi.MXFP4_QUANT_RHT_COL, 0x1357),
                              (w.cuda(), 520, 200, 200, *bw[0], *bw[1], abi.MXFP4_QUANT_2D_BLOCKS)], True)
    torch.cuda.synchronize()
    assert abi.mxfp4_last_device_error() == abi.MXFP4_OK
    for got, want in zip([*bx[0], *bx[1]], sx):
        assert torch.equal(got.cpu(), want.cpu())
    for got, want in zip([*bw[0], *bw[1]], sw):
        assert torch.equal(got.cpu(), want.cpu())


# --- the gradient recipe with `use_sr`: transformed col blob, stochastic rounding ---------

def check_rht_sr_full(x_cpu, outs, layout, signs, seed, what):
    xb = workloads.bf16_bits(x_cpu)
    tc = layout == abi.MXFP4_SCALE_TC
    rq, rs = oracle.quantize_row_sr(xb, seed)
    assert_bytes_equal(outs[0].cpu().numpy(), rq, f"{what} row q")
    assert_bytes_equal(outs[1].cpu().numpy().reshape(-1), (oracle.scale_to_tc(rs) if tc else rs).reshape(-1),
                       f"{what} row s")
    cq, cs = oracle.quantize_col_rht_sr(xb, signs, seed)
    assert_bytes_equal(outs[2].cpu().numpy(), cq, f"{what} col q")
    assert_bytes_equal(outs[3].cpu().numpy().reshape(-1), (oracle.scale_to_tc(cs) if tc else cs).reshape(-1),
                       f"{what} col s")


@pytest.mark.parametrize("M,K,ldx", [(1, 8, 8), (40, 40, 40), (130, 200, 200), (257, 33, 40), (640, 384, 384),
                                     (4600, 256, 256)])
@pytest.mark.parametrize("signs,seed", [(0xA5C3, 7), (0x8001, 0x9E3779B97F4A7C15)])
def test_rht_sr_ragged_shapes(M, K, ldx, signs, seed):
    # Row blob as the stochastically rounded dual quantizer, col blob as the oracle's
    # transformed and stochastically rounded columns, byte for byte.
    x = _rht_input(M, K, 7 * M + K)
    for layout in LAYOUTS:
        wide = torch.zeros((M, ldx), dtype=torch.bfloat16)
        wide[:, :K] = x
        outs = abi.quantize(wide.cuda()[:, :K], dual=True, layout=layout, rht_signs=signs, sr_seed=seed)
        torch.cuda.synchronize()
        assert abi.mxfp4_last_device_error() == abi.MXFP4_OK
        check_rht_sr_full(x, outs, layout, signs, seed, f"rht+sr {M}x{K}")


def test_rht_sr_every_bf16_pattern_below_overflow():
    b = np.arange(0x10000, dtype=np.uint32).astype(np.uint16)
    b = np.where((b & 0x7F80) < (200 << 7), b, 0).astype(np.uint16)
    rng = np.random.default_rng(17)
    x = _bits_to_bf16(b[rng.permutation(b.size)].reshape(256, 256))
    outs = abi.quantize(x.cuda(), dual=True, layout=abi.MXFP4_SCALE_TC, rht_signs=0x1234, sr_seed=99)
    torch.cuda.synchronize()
    check_rht_sr_full(x, outs, abi.MXFP4_SCALE_TC, 0x1234, 99, "rht+sr all patterns")


def test_rht_sr_seed_behaviour():
    # Same seed: identical bytes; another seed: other elements, the same scales, which are
    # the round-to-nearest transformed ones.
    x = workloads.normal((384, 640), 1.0, 79).cuda()
    a = abi.quantize(x, dual=True, rht_signs=0xA5C3, sr_seed=5)
    b = abi.quantize(x, dual=True, rht_signs=0xA5C3, sr_seed=5)
    c = abi.quantize(x, dual=True, rht_signs=0xA5C3, sr_seed=6)
    n = abi.quantize(x, dual=True, rht_signs=0xA5C3)
    torch.cuda.synchronize()
    for u, v in zip(a, b):
        assert torch.equal(u, v)
    assert not torch.equal(a[2], c[2])
    assert torch.equal(a[1], n[1]) and torch.equal(a[3], n[3])


def test_rht_sr_flux_dy_sampled():
    # The single-stream block's two gradients dY [4608, 21504] and [4608, 3072] in the
    # launch configuration of the backward step, on sampled rows and columns at their true
    # positions.
    from parity import gather_tc_rows
    seed = 4242
    for li in (0, 1):
        dy = workloads.FLUX_SINGLE_BLOCK.tensors(li)["dY"]
        outs = abi.quantize(dy.cuda(), dual=True, layout=abi.MXFP4_SCALE_TC, rht_signs=0xA5C3, sr_seed=seed)
        torch.cuda.synchronize()
        assert abi.mxfp4_last_device_error() == abi.MXFP4_OK
        xb = workloads.bf16_bits(dy)
        M, K = xb.shape
        rng = np.random.default_rng(11 + li)
        rows = np.unique(np.concatenate([rng.choice(M, 16, replace=False), [0, M - 1]]))
        cols = np.unique(np.concatenate([rng.choice(K, 16, replace=False), [0, K - 1]]))
        rq, rs = oracle.quantize_row_sr(np.ascontiguousarray(xb[rows]), seed, row_ids=rows)
        assert_bytes_equal(outs[0][torch.as_tensor(rows, device="cuda")].cpu().numpy(), rq, f"dY{li} row q")
        assert_bytes_equal(gather_tc_rows(outs[1].cpu().numpy(), rows, rs.shape[1]), rs, f"dY{li} row s")
        cq, cs = oracle.quantize_col_rht_sr(np.ascontiguousarray(xb[:, cols]), 0xA5C3, seed, col_ids=cols)
        assert_bytes_equal(outs[2][torch.as_tensor(cols, device="cuda")].cpu().numpy(), cq, f"dY{li} col q")
        assert_bytes_equal(gather_tc_rows(outs[3].cpu().numpy(), cols, cs.shape[1]), cs, f"dY{li} col s")

