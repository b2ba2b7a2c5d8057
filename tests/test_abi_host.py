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
    G = abi.GemmTask
    g_ok = G(16, 32, 48, 64, 4, 4, 4, 80, 4, 0)
    garr = (G * 5)(*([g_ok] * 5))
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
    assert lib.mxfp4_gemm(0x10000, 0x20000, 0x30000, 0x40000, 4, 4, 4, 0x50000, 4, 0, None) in bad
    assert lib.mxfp4_gemm_bias(0x10000, 0x20000, 0x30000, 0x40000, 4, 4, 4, 0x60000, 0x50000, 4, 0, None) in bad
    assert lib.mxfp4_fp8_quantize_tw(0x10000, 4, 8, 8, 0x20000, None, 0x30000, 0x30004, None) in bad
    assert lib.mxfp4_fp8_gemm(0x10000, 0x20000, 0x30000, 0x40000, 4, 4, 4, 0x50000, 4, 0, None) in bad
    assert lib.mxfp4_last_device_error(None) in bad


def test_status_strings(lib):
    for code in range(6):
        assert abi.status_string(code).startswith("MXFP4_")
    assert "unknown" in abi.status_string(99)
