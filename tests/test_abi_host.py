"""Host-side checks of the C ABI that need no GPU: the library loads, exports every
function include/mxfp4.h declares, and rejects bad arguments before touching a device."""
import ctypes
import os
import re
import subprocess

import pytest

from mxfp4_block_scaled_quantize_gb300 import abi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    return abi.load()


def declared_functions():
    with open(os.path.join(ROOT, "include", "mxfp4.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mxfp4_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_abi():
    assert declared_functions() == sorted(abi.EXPORTED)


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", abi.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (mxfp4_[a-z_0-9]+)$", out, flags=re.M))
    for name in declared_functions():
        assert name in exported, name
        assert getattr(lib, name) is not None


def test_sizes_match_the_shape_contract(lib):
    # [4608, 3072] row blob and col blob, plain and tensor-core scale layouts
    assert abi.mxfp4_quantize_sizes(4608, 3072, abi.MXFP4_SCALE_PLAIN) == (4608 * 1536, 4608 * 96)
    assert abi.mxfp4_quantize_sizes(3072, 4600, abi.MXFP4_SCALE_PLAIN) == (3072 * 2304, 3072 * 144)
    assert abi.mxfp4_quantize_sizes(4600, 3072, abi.MXFP4_SCALE_TC) == (4600 * 1536, 4608 * 96)
    assert abi.mxfp4_quantize_sizes(1, 1, abi.MXFP4_SCALE_TC) == (64, 128 * 4)
    for bad in ((0, 1, 0), (1, 0, 0), (-5, 8, 1), (8, 8, 2)):
        with pytest.raises(abi.Mxfp4Error) as e:
            abi.mxfp4_quantize_sizes(*bad)
        assert e.value.status == abi.MXFP4_ERR_INVALID_ARG


def test_argument_checks_precede_any_device_use(lib):
    vp = ctypes.c_void_p
    assert lib.mxfp4_quantize(None, 4, 4, 8, None, None, 0, None) == abi.MXFP4_ERR_INVALID_ARG
    assert lib.mxfp4_quantize(16, 4, 16, 8, 32, 48, 0, None) == abi.MXFP4_ERR_INVALID_ARG  # ldx < K
    assert lib.mxfp4_quantize(18, 4, 8, 8, 32, 48, 0, None) == abi.MXFP4_ERR_MISALIGNED
    assert lib.mxfp4_quantize(16, 4, 6, 6, 32, 48, 0, None) == abi.MXFP4_ERR_MISALIGNED
    assert lib.mxfp4_quantize_dual(16, 4, 8, 8, 32, 48, None, 64, 1, None) == abi.MXFP4_ERR_INVALID_ARG
    assert lib.mxfp4_quantize_dual_sr(16, 4, 8, 8, 32, 48, None, 64, 1, 7, None) == abi.MXFP4_ERR_INVALID_ARG
    assert lib.mxfp4_quantize_dual_sr(18, 4, 8, 8, 32, 48, 64, 80, 1, 7, None) == abi.MXFP4_ERR_MISALIGNED
    assert lib.mxfp4_gemm(16, 32, 48, 64, 4, 4, 4, 80, 2, 0, None) == abi.MXFP4_ERR_INVALID_ARG
    assert lib.mxfp4_gemm(16, 32, 48, 64, 4, 4, 4, 88, 4, 0, None) == abi.MXFP4_ERR_MISALIGNED
    assert lib.mxfp4_selftest_bounded_wait(0, None) == abi.MXFP4_ERR_INVALID_ARG
    # batch: task count, task array, and each task's own checks
    T = abi.QuantizeTask
    good = T(16, 4, 8, 8, 32, 48, 64, 80)
    arr = (T * 5)(*([good] * 5))
    assert lib.mxfp4_quantize_batch(0, arr, 1, 1, None) == abi.MXFP4_ERR_INVALID_ARG
    assert lib.mxfp4_quantize_batch(5, arr, 1, 1, None) == abi.MXFP4_ERR_INVALID_ARG
    assert lib.mxfp4_quantize_batch(1, None, 1, 1, None) == abi.MXFP4_ERR_INVALID_ARG
    bad = (T * 2)(good, T(16, 4, 8, 8, 32, 48, None, 80))          # dual without q_col
    assert lib.mxfp4_quantize_batch(2, bad, 1, 1, None) == abi.MXFP4_ERR_INVALID_ARG
    bad = (T * 2)(good, T(18, 4, 8, 8, 32, 48, 64, 80))            # x not 16-byte aligned
    assert lib.mxfp4_quantize_batch(2, bad, 1, 1, None) == abi.MXFP4_ERR_MISALIGNED
    assert lib.mxfp4_quantize_batch(1, arr, 1, 2, None) == abi.MXFP4_ERR_INVALID_ARG  # layout
    bad = (T * 2)(good, T(16, 4, 8, 8, 32, 48, 64, 80, 4))         # unknown flag bit
    assert lib.mxfp4_quantize_batch(2, bad, 1, 1, None) == abi.MXFP4_ERR_INVALID_ARG
    bad = (T * 2)(good, T(16, 4, 8, 8, 32, 48, 64, 80, 3))         # 2-D and transform together
    assert lib.mxfp4_quantize_batch(2, bad, 1, 1, None) == abi.MXFP4_ERR_INVALID_ARG
    bad = (T * 1)(T(16, 4, 8, 8, 32, 48, 64, 80, 2, 7))            # transform without a col blob
    assert lib.mxfp4_quantize_batch(1, bad, 0, 1, None) == abi.MXFP4_ERR_INVALID_ARG
    assert lib.mxfp4_quantize_dual_rht(16, 4, 8, 8, 32, 48, None, 64, 1, 7, None) == abi.MXFP4_ERR_INVALID_ARG
    assert lib.mxfp4_quantize_dual_rht_sr(16, 4, 8, 8, 32, 48, None, 64, 1, 7, 9, None) == abi.MXFP4_ERR_INVALID_ARG
    nr = [16, 32, 4, 1, 48, 64, 80, 96, 112, 128, 144, 160, 176, 1, None, None]
    assert lib.mxfp4_quantize_dual_qk_norm_rope_bwd(*nr[:3], 0, *nr[4:]) == abi.MXFP4_ERR_INVALID_ARG  # H
    bad = list(nr)
    bad[1] = None                                                    # no mixed_qkv
    assert lib.mxfp4_quantize_dual_qk_norm_rope_bwd(*bad) == abi.MXFP4_ERR_INVALID_ARG
    bad = list(nr)
    bad[7] = 100                                                     # cos table not 16-byte aligned
    assert lib.mxfp4_quantize_dual_qk_norm_rope_bwd(*bad) == abi.MXFP4_ERR_MISALIGNED
    assert lib.mxfp4_quantize_dual_rht_sr(16, 4, 8, 8, 32, 48, 64, 80, 3, 7, 9, None) == abi.MXFP4_ERR_INVALID_ARG
    assert lib.mxfp4_quantize_dual_2d(16, 4, 8, 8, 32, 48, None, 64, 1, None) == abi.MXFP4_ERR_INVALID_ARG
    assert lib.mxfp4_quantize_dual_2d(18, 4, 8, 8, 32, 48, 64, 80, 1, None) == abi.MXFP4_ERR_MISALIGNED
    ok = (16, 32, 48, 64, 300, 200, 264, None, 80, 200, 96, 112, 128, 144, None)
    bad = list(ok)
    bad[9] = 204                                                     # ldc not a multiple of 8
    assert lib.mxfp4_gemm_quantize(*bad) == abi.MXFP4_ERR_MISALIGNED
    bad = list(ok)
    bad[10] = None                                                   # no row blob
    assert lib.mxfp4_gemm_quantize(*bad) == abi.MXFP4_ERR_INVALID_ARG
    bad = list(ok)
    bad[13] = None                                                   # q_col without s_col
    assert lib.mxfp4_gemm_quantize(*bad) == abi.MXFP4_ERR_INVALID_ARG
    bad = list(ok)
    bad[11] = 120                                                    # s_row not 16-byte aligned
    assert lib.mxfp4_gemm_quantize(*bad) == abi.MXFP4_ERR_MISALIGNED
    T2 = abi.QuantizeTask
    amax_dual = (T2 * 1)(T2(16, 4, 8, 8, 32, 48, 64, 80, 0, 0, 96))     # amax with the dual quantizer
    assert lib.mxfp4_quantize_batch(1, amax_dual, 1, 1, None) == abi.MXFP4_ERR_INVALID_ARG
    amax_odd = (T2 * 1)(T2(16, 4, 8, 8, 32, 48, None, None, 0, 0, 98))  # amax not 4-byte aligned
    assert lib.mxfp4_quantize_batch(1, amax_odd, 0, 1, None) == abi.MXFP4_ERR_MISALIGNED
    G = abi.GemmTask
    g_ok = G(16, 32, 48, 64, 4, 4, 4, 80, 4, 0)
    garr = (G * 5)(*([g_ok] * 5))
    assert lib.mxfp4_linear_step_host_pipelined(0, None, None, 0, None) == abi.MXFP4_ERR_INVALID_ARG
    assert lib.mxfp4_linear_pipelined_workspace_bytes(1, None, None) == abi.MXFP4_ERR_INVALID_ARG
    assert lib.mxfp4_gemm_set_tile_policy(3) == abi.MXFP4_ERR_INVALID_ARG
    assert lib.mxfp4_gemm_set_tile_policy(-1) == abi.MXFP4_ERR_INVALID_ARG
    assert lib.mxfp4_gemm_set_tile_policy(abi.MXFP4_TILES_AUTO) == abi.MXFP4_OK
    assert lib.mxfp4_gemm_batch(0, garr, None) == abi.MXFP4_ERR_INVALID_ARG
    assert lib.mxfp4_gemm_batch(5, garr, None) == abi.MXFP4_ERR_INVALID_ARG
    assert lib.mxfp4_gemm_batch(1, None, None) == abi.MXFP4_ERR_INVALID_ARG
    gbad = (G * 2)(g_ok, G(16, 32, 48, 64, 4, 4, 4, 80, 2, 0))     # ldc < N
    assert lib.mxfp4_gemm_batch(2, gbad, None) == abi.MXFP4_ERR_INVALID_ARG
    gbad = (G * 2)(g_ok, G(16, 32, 48, 64, 4, 4, 4, 88, 4, 0))     # c not 16-byte aligned
    assert lib.mxfp4_gemm_batch(2, gbad, None) == abi.MXFP4_ERR_MISALIGNED
    gbad = (G * 1)(G(16, 32, 48, 64, 4, 4, 4, 80, 4, 7))           # out dtype
    assert lib.mxfp4_gemm_batch(1, gbad, None) == abi.MXFP4_ERR_INVALID_ARG
    gbad = (G * 2)(g_ok, G(16, 32, 48, 64, 4, 4, 4, 80, 4, 0, 104))  # bias not 16-byte aligned
    assert lib.mxfp4_gemm_batch(2, gbad, None) == abi.MXFP4_ERR_MISALIGNED
    # the bias entry point: bias required and 16-byte aligned, then the GEMM's own checks
    assert lib.mxfp4_gemm_bias(16, 32, 48, 64, 4, 4, 4, None, 80, 4, 0, None) == abi.MXFP4_ERR_INVALID_ARG
    assert lib.mxfp4_gemm_bias(16, 32, 48, 64, 4, 4, 4, 104, 80, 4, 0, None) == abi.MXFP4_ERR_MISALIGNED
    assert lib.mxfp4_gemm_bias(16, 32, 48, 64, 4, 4, 4, 96, 80, 2, 0, None) == abi.MXFP4_ERR_INVALID_ARG


def test_fp8_argument_checks_precede_any_device_use(lib):
    # quantize: input, at least one output copy, scalar outputs, alignment
    assert lib.mxfp4_fp8_quantize_tw(16, 4, 8, 8, None, None, 64, 68, None) == abi.MXFP4_ERR_INVALID_ARG
    assert lib.mxfp4_fp8_quantize_tw(16, 4, 8, 8, 32, None, None, 68, None) == abi.MXFP4_ERR_INVALID_ARG
    assert lib.mxfp4_fp8_quantize_tw(16, 4, 8, 6, 32, None, 64, 68, None) == abi.MXFP4_ERR_INVALID_ARG
    assert lib.mxfp4_fp8_quantize_tw(16, 4, 8, 12, 32, None, 64, 68, None) == abi.MXFP4_ERR_MISALIGNED
    assert lib.mxfp4_fp8_quantize_tw(16, 4, 8, 8, 40, None, 64, 68, None) == abi.MXFP4_ERR_MISALIGNED
    assert lib.mxfp4_fp8_quantize_tw(16, 4, 8, 8, 32, 48, 66, 68, None) == abi.MXFP4_ERR_MISALIGNED
    Q = abi.Fp8QuantizeTask
    q_ok = Q(16, 4, 8, 8, 32, None, 64, 68)
    qarr = (Q * 5)(*([q_ok] * 5))
    assert lib.mxfp4_fp8_quantize_tw_batch(0, qarr, None) == abi.MXFP4_ERR_INVALID_ARG
    assert lib.mxfp4_fp8_quantize_tw_batch(5, qarr, None) == abi.MXFP4_ERR_INVALID_ARG
    qbad = (Q * 2)(q_ok, Q(16, 4, 8, 8, None, None, 64, 68))      # no output copy
    assert lib.mxfp4_fp8_quantize_tw_batch(2, qbad, None) == abi.MXFP4_ERR_INVALID_ARG
    qbad = (Q * 2)(q_ok, Q(16, 4, 8, 8, 40, None, 64, 68))        # q_row not 16-byte aligned
    assert lib.mxfp4_fp8_quantize_tw_batch(2, qbad, None) == abi.MXFP4_ERR_MISALIGNED
    # GEMM: operands, scales, output pitch, dtype, alignment
    assert lib.mxfp4_fp8_gemm(16, None, 48, 64, 4, 4, 4, 80, 4, 0, None) == abi.MXFP4_ERR_INVALID_ARG
    assert lib.mxfp4_fp8_gemm(16, 32, 48, 64, 4, 4, 4, 80, 2, 0, None) == abi.MXFP4_ERR_INVALID_ARG
    assert lib.mxfp4_fp8_gemm(16, 32, 48, 64, 4, 4, 4, 80, 4, 3, None) == abi.MXFP4_ERR_INVALID_ARG
    assert lib.mxfp4_fp8_gemm(16, 34, 48, 64, 4, 4, 4, 80, 4, 0, None) == abi.MXFP4_ERR_MISALIGNED
    assert lib.mxfp4_fp8_gemm(24, 32, 48, 64, 4, 4, 4, 80, 4, 0, None) == abi.MXFP4_ERR_MISALIGNED
    G = abi.Fp8GemmTask
    g_ok = G(16, 32, 48, 64, 4, 4, 4, 80, 4, 0)
    garr = (G * 5)(*([g_ok] * 5))
    assert lib.mxfp4_fp8_gemm_batch(0, garr, None) == abi.MXFP4_ERR_INVALID_ARG
    assert lib.mxfp4_fp8_gemm_batch(5, garr, None) == abi.MXFP4_ERR_INVALID_ARG
    gbad = (G * 2)(g_ok, G(16, 32, 48, 64, 4, 4, 4, 88, 4, 0))
    assert lib.mxfp4_fp8_gemm_batch(2, gbad, None) == abi.MXFP4_ERR_MISALIGNED


def test_no_usable_device_fails_loudly(lib):
    # Well-formed calls on a host without a CUDA device return an error status (no
    # fallback path, nothing dereferenced: the device gate comes before any launch).
    import torch
    if torch.cuda.is_available():
        pytest.skip("a CUDA device is present")
    bad = (abi.MXFP4_ERR_CUDA, abi.MXFP4_ERR_UNSUPPORTED_DEVICE)
    assert lib.mxfp4_quantize(0x10000, 4, 8, 8, 0x20000, 0x30000, 1, None) in bad
    assert lib.mxfp4_quantize_dual(0x10000, 4, 8, 8, 0x20000, 0x30000, 0x40000, 0x50000, 1, None) in bad
    assert lib.mxfp4_quantize_dual_sr(0x10000, 4, 8, 8, 0x20000, 0x30000, 0x40000, 0x50000, 1, 7, None) in bad
    assert lib.mxfp4_quantize_dual_2d(0x10000, 4, 8, 8, 0x20000, 0x30000, 0x40000, 0x50000, 1, None) in bad
    assert lib.mxfp4_quantize_dual_rht(0x10000, 4, 8, 8, 0x20000, 0x30000, 0x40000, 0x50000, 1, 7, None) in bad
    assert lib.mxfp4_quantize_dual_rht_sr(0x10000, 4, 8, 8, 0x20000, 0x30000, 0x40000, 0x50000, 1, 7, 9,
                                          None) in bad
    assert lib.mxfp4_quantize_dual_qk_norm_rope_bwd(0x10000, 0x20000, 4, 1, 0x30000, 0x40000, 0x50000, 0x60000,
                                                    0x70000, 0x80000, 0x90000, 0xA0000, 0xB0000, 1, None,
                                                    None) in bad
    assert lib.mxfp4_gemm(0x10000, 0x20000, 0x30000, 0x40000, 4, 4, 4, 0x50000, 4, 0, None) in bad
    assert lib.mxfp4_gemm_bias(0x10000, 0x20000, 0x30000, 0x40000, 4, 4, 4, 0x60000, 0x50000, 4, 0, None) in bad
    assert lib.mxfp4_gemm_quantize(0x10000, 0x20000, 0x30000, 0x40000, 4, 8, 4, None, 0x50000, 8, 0x60000, 0x70000,
                                   None, None, None) in bad
    assert lib.mxfp4_fp8_quantize_tw(0x10000, 4, 8, 8, 0x20000, None, 0x30000, 0x30004, None) in bad
    assert lib.mxfp4_fp8_gemm(0x10000, 0x20000, 0x30000, 0x40000, 4, 4, 4, 0x50000, 4, 0, None) in bad
    task = (abi.LinearHostTask * 1)(abi.LinearHostTask(0x1000, 0x2000, 0, 0x4000, 0, 0, 4, 8, 16, 0, 0))
    assert lib.mxfp4_linear_step_host(1, task, 0x100000, 1 << 20, None) in bad
    assert lib.mxfp4_last_device_error(None) in bad


def test_status_strings(lib):
    for code in range(7):
        assert abi.status_string(code).startswith("MXFP4_")
    assert "unknown" in abi.status_string(99)


def _host_task(M=4, N=8, K=16, train=0, od=0, x=0x1000, w=0x2000, dy=0x3000, y=0x4000, dx=0x5000, dw=0x6000):
    return abi.LinearHostTask(x, w, dy, y, dx, dw, M, N, K, train, od)


def test_linear_workspace_bytes(lib):
    # Forward-only M 4, N 8, K 16, bf16 out: device X (4 x 16 bf16 = 128 B), W (256 B), X row
    # blob (4 x 64 B codes; 128 padded rows x 4 scale bytes), W row blob (8 x 64 B; 512 B),
    # Y (4 x 8 bf16 = 64 B), every piece rounded up to 256 bytes.
    n = ctypes.c_size_t()
    arr = (abi.LinearHostTask * 1)(_host_task())
    assert lib.mxfp4_linear_workspace_bytes(1, arr, ctypes.byref(n)) == abi.MXFP4_OK
    assert n.value == 256 + 256 + 256 + 512 + 512 + 512 + 256
    # training adds dY (4 x 8 bf16), the col blobs of X, W and both blobs of dY, dX, dW;
    # K = 12 is padded to a row pitch of 16 elements for the device copies of X and W.
    arr = (abi.LinearHostTask * 1)(_host_task(M=4, N=8, K=12, train=1))
    assert lib.mxfp4_linear_workspace_bytes(1, arr, ctypes.byref(n)) == abi.MXFP4_OK
    fwd = 256 + 256 + 256 + 512 + 512 + 512 + 256
    dy = 256
    x_col = 12 * 64 + 128 * 4          # [12, Mp/2 = 64] codes, 128 x (Mp/32 = 4) scales
    w_col = 12 * 64 + 128 * 4
    dy_row = 4 * 64 + 128 * 4
    dy_col = 8 * 64 + 128 * 4
    dxdw = 256 + 256                   # 4 x 12 and 8 x 12 bf16, each under 256 bytes
    r = lambda b: (b + 255) // 256 * 256
    want = fwd + dy + r(12 * 64) + 512 + r(12 * 64) + 512 + r(4 * 64) + 512 + r(8 * 64) + 512 + dxdw
    assert n.value == want
    # two tasks: the sum of both
    arr2 = (abi.LinearHostTask * 2)(_host_task(), _host_task(M=4, N=8, K=12, train=1))
    assert lib.mxfp4_linear_workspace_bytes(2, arr2, ctypes.byref(n)) == abi.MXFP4_OK
    assert n.value == fwd + want


def test_linear_step_host_argument_checks(lib):
    T = abi.LinearHostTask
    ok = (T * 5)(*([_host_task()] * 5))
    n = ctypes.c_size_t()
    assert lib.mxfp4_linear_workspace_bytes(0, ok, ctypes.byref(n)) == abi.MXFP4_ERR_INVALID_ARG
    assert lib.mxfp4_linear_workspace_bytes(5, ok, ctypes.byref(n)) == abi.MXFP4_ERR_INVALID_ARG
    assert lib.mxfp4_linear_workspace_bytes(1, ok, None) == abi.MXFP4_ERR_INVALID_ARG
    for bad in (_host_task(M=0), _host_task(od=3), _host_task(train=2)):
        arr = (T * 2)(_host_task(), bad)
        assert lib.mxfp4_linear_workspace_bytes(2, arr, ctypes.byref(n)) == abi.MXFP4_ERR_INVALID_ARG
        assert lib.mxfp4_linear_step_host(2, arr, 0x100000, 1 << 20, None) == abi.MXFP4_ERR_INVALID_ARG
    # the size query reads shapes only; the step needs every host buffer of its mode
    for bad in (_host_task(x=0), _host_task(y=0), _host_task(train=1, dy=0), _host_task(train=1, dw=0)):
        arr = (T * 2)(_host_task(), bad)
        assert lib.mxfp4_linear_workspace_bytes(2, arr, ctypes.byref(n)) == abi.MXFP4_OK
        assert lib.mxfp4_linear_step_host(2, arr, 0x100000, 1 << 20, None) == abi.MXFP4_ERR_INVALID_ARG
    one = (T * 1)(_host_task())
    assert lib.mxfp4_linear_step_host(1, one, None, 1 << 20, None) == abi.MXFP4_ERR_INVALID_ARG
    assert lib.mxfp4_linear_step_host(1, one, 0x100000, 100, None) == abi.MXFP4_ERR_INVALID_ARG   # too small
    assert lib.mxfp4_linear_step_host(1, one, 0x100010, 1 << 20, None) == abi.MXFP4_ERR_MISALIGNED
