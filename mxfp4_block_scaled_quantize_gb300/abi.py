"""Python binding of the C ABI in include/mxfp4.h (argument marshalling only).

Every function named like a C entry point forwards to it through ctypes; buffers may be
given as torch CUDA tensors or as raw device addresses (int).  PyTorch serves only as the
allocator and the source of the current stream.  Nothing here computes: if the CUDA
library is missing, loading raises -- there is no fallback path.
"""
import ctypes
import os
from typing import Optional, Tuple

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libmxfp4_gb300.so")

MXFP4_OK = 0
MXFP4_ERR_INVALID_ARG = 1
MXFP4_ERR_MISALIGNED = 2
MXFP4_ERR_UNSUPPORTED_DEVICE = 3
MXFP4_ERR_CUDA = 4
MXFP4_ERR_TIMEOUT = 5
MXFP4_ERR_NONFINITE = 6

MXFP4_SCALE_PLAIN = 0
MXFP4_SCALE_TC = 1

MXFP4_OUT_BF16 = 0
MXFP4_OUT_F32 = 1

MXFP4_MAX_BATCH = 4

MXFP4_TILES_AUTO = 0
MXFP4_TILES_NARROW = 1
MXFP4_TILES_WIDE = 2


class GemmTask(ctypes.Structure):
    """mxfp4_gemm_task of include/mxfp4.h."""
    _fields_ = [("a_q", ctypes.c_void_p), ("a_s", ctypes.c_void_p), ("b_q", ctypes.c_void_p),
                ("b_s", ctypes.c_void_p), ("M", ctypes.c_int64), ("N", ctypes.c_int64),
                ("K", ctypes.c_int64), ("c", ctypes.c_void_p), ("ldc", ctypes.c_int64),
                ("out_dtype", ctypes.c_int), ("bias", ctypes.c_void_p)]


class QuantizeTask(ctypes.Structure):
    """mxfp4_quantize_task of include/mxfp4.h."""
    _fields_ = [("x", ctypes.c_void_p), ("rows", ctypes.c_int64), ("k", ctypes.c_int64),
                ("ldx", ctypes.c_int64), ("q_row", ctypes.c_void_p), ("s_row", ctypes.c_void_p),
                ("q_col", ctypes.c_void_p), ("s_col", ctypes.c_void_p), ("flags", ctypes.c_int32),
                ("rht_signs", ctypes.c_uint32), ("amax", ctypes.c_void_p)]


MXFP4_QUANT_2D_BLOCKS = 1
MXFP4_QUANT_RHT_COL = 2

class Fp8QuantizeTask(ctypes.Structure):
    """mxfp4_fp8_quantize_task of include/mxfp4.h."""
    _fields_ = [("x", ctypes.c_void_p), ("M", ctypes.c_int64), ("K", ctypes.c_int64), ("ldx", ctypes.c_int64),
                ("q_row", ctypes.c_void_p), ("q_col", ctypes.c_void_p), ("amax", ctypes.c_void_p),
                ("scale_inv", ctypes.c_void_p), ("amax_given", ctypes.c_int32)]


class Fp8GemmTask(ctypes.Structure):
    """mxfp4_fp8_gemm_task of include/mxfp4.h."""
    _fields_ = [("a", ctypes.c_void_p), ("a_scale_inv", ctypes.c_void_p), ("b", ctypes.c_void_p),
                ("b_scale_inv", ctypes.c_void_p), ("M", ctypes.c_int64), ("N", ctypes.c_int64),
                ("K", ctypes.c_int64), ("c", ctypes.c_void_p), ("ldc", ctypes.c_int64),
                ("out_dtype", ctypes.c_int)]


class LinearHostTask(ctypes.Structure):
    """mxfp4_linear_host_task of include/mxfp4.h."""
    _fields_ = [("x", ctypes.c_void_p), ("w", ctypes.c_void_p), ("dy", ctypes.c_void_p),
                ("y", ctypes.c_void_p), ("dx", ctypes.c_void_p), ("dw", ctypes.c_void_p),
                ("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("train", ctypes.c_int32), ("out_dtype", ctypes.c_int)]


EXPORTED = (
    "mxfp4_quantize_sizes",
    "mxfp4_quantize",
    "mxfp4_quantize_dual",
    "mxfp4_quantize_dual_sr",
    "mxfp4_quantize_dual_2d",
    "mxfp4_quantize_dual_rht",
    "mxfp4_quantize_dual_rht_sr",
    "mxfp4_quantize_dual_qk_norm_rope_bwd",
    "mxfp4_quantize_batch",
    "mxfp4_gemm",
    "mxfp4_gemm_bias",
    "mxfp4_gemm_quantize",
    "mxfp4_gemm_batch",
    "mxfp4_gemm_set_tile_policy",
    "mxfp4_fp8_quantize_tw",
    "mxfp4_fp8_quantize_tw_batch",
    "mxfp4_fp8_gemm",
    "mxfp4_fp8_gemm_batch",
    "mxfp4_linear_workspace_bytes",
    "mxfp4_linear_step_host",
    "mxfp4_linear_pipelined_workspace_bytes",
    "mxfp4_linear_step_host_pipelined",
    "mxfp4_linear_host_wait",
    "mxfp4_last_device_error",
    "mxfp4_selftest_bounded_wait",
    "mxfp4_status_string",
)


class Mxfp4Error(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)}")


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads the CUDA library (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"CUDA library {path} not found: build it first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    i64, vp, i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
    lib.mxfp4_quantize_sizes.argtypes = [i64, i64, i32, ctypes.POINTER(ctypes.c_size_t),
                                         ctypes.POINTER(ctypes.c_size_t)]
    lib.mxfp4_quantize.argtypes = [vp, i64, i64, i64, vp, vp, i32, vp]
    lib.mxfp4_quantize_dual.argtypes = [vp, i64, i64, i64, vp, vp, vp, vp, i32, vp]
    lib.mxfp4_quantize_dual_sr.argtypes = [vp, i64, i64, i64, vp, vp, vp, vp, i32, ctypes.c_uint64, vp]
    lib.mxfp4_quantize_dual_2d.argtypes = [vp, i64, i64, i64, vp, vp, vp, vp, i32, vp]
    lib.mxfp4_quantize_dual_rht.argtypes = [vp, i64, i64, i64, vp, vp, vp, vp, i32, ctypes.c_uint32, vp]
    lib.mxfp4_quantize_dual_rht_sr.argtypes = [vp, i64, i64, i64, vp, vp, vp, vp, i32, ctypes.c_uint32,
                                               ctypes.c_uint64, vp]
    lib.mxfp4_quantize_dual_qk_norm_rope_bwd.argtypes = [vp, vp, i64, i64, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32,
                                                         vp, vp]
    lib.mxfp4_quantize_batch.argtypes = [i32, ctypes.POINTER(QuantizeTask), i32, i32, vp]
    lib.mxfp4_gemm.argtypes = [vp, vp, vp, vp, i64, i64, i64, vp, i64, i32, vp]
    lib.mxfp4_gemm_bias.argtypes = [vp, vp, vp, vp, i64, i64, i64, vp, vp, i64, i32, vp]
    lib.mxfp4_gemm_batch.argtypes = [i32, ctypes.POINTER(GemmTask), vp]
    lib.mxfp4_gemm_set_tile_policy.argtypes = [i32]
    lib.mxfp4_gemm_quantize.argtypes = [vp, vp, vp, vp, i64, i64, i64, vp, vp, i64, vp, vp, vp, vp, vp]
    lib.mxfp4_fp8_quantize_tw.argtypes = [vp, i64, i64, i64, vp, vp, vp, vp, vp]
    lib.mxfp4_fp8_quantize_tw_batch.argtypes = [i32, ctypes.POINTER(Fp8QuantizeTask), vp]
    lib.mxfp4_fp8_gemm.argtypes = [vp, vp, vp, vp, i64, i64, i64, vp, i64, i32, vp]
    lib.mxfp4_fp8_gemm_batch.argtypes = [i32, ctypes.POINTER(Fp8GemmTask), vp]
    lib.mxfp4_linear_workspace_bytes.argtypes = [i32, ctypes.POINTER(LinearHostTask),
                                                 ctypes.POINTER(ctypes.c_size_t)]
    lib.mxfp4_linear_step_host.argtypes = [i32, ctypes.POINTER(LinearHostTask), vp, ctypes.c_size_t, vp]
    lib.mxfp4_linear_pipelined_workspace_bytes.argtypes = [i32, ctypes.POINTER(LinearHostTask),
                                                           ctypes.POINTER(ctypes.c_size_t)]
    lib.mxfp4_linear_step_host_pipelined.argtypes = [i32, ctypes.POINTER(LinearHostTask), vp, ctypes.c_size_t, vp]
    lib.mxfp4_linear_host_wait.argtypes = [vp]
    lib.mxfp4_last_device_error.argtypes = [vp]
    lib.mxfp4_selftest_bounded_wait.argtypes = [i64, vp]
    lib.mxfp4_status_string.argtypes = [i32]
    lib.mxfp4_status_string.restype = ctypes.c_char_p
    for name in EXPORTED[:-1]:
        getattr(lib, name).restype = i32
    _lib = lib
    return lib


def _ptr(buf) -> Optional[int]:
    if buf is None:
        return None
    if isinstance(buf, int):
        return buf
    return buf.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, what: str) -> None:
    if status != MXFP4_OK:
        raise Mxfp4Error(status, what)


def status_string(status: int) -> str:
    return load().mxfp4_status_string(int(status)).decode()


# ---------------------------------------------------------------------------------------
# the C entry points
# ---------------------------------------------------------------------------------------
def mxfp4_quantize_sizes(rows: int, k: int, layout: int = MXFP4_SCALE_TC) -> Tuple[int, int]:
    q = ctypes.c_size_t()
    s = ctypes.c_size_t()
    _check(load().mxfp4_quantize_sizes(rows, k, layout, ctypes.byref(q), ctypes.byref(s)),
           "mxfp4_quantize_sizes")
    return q.value, s.value


def mxfp4_quantize(x, M, K, ldx, q_row, s_row, layout=MXFP4_SCALE_TC, stream=None) -> None:
    _check(load().mxfp4_quantize(_ptr(x), M, K, ldx, _ptr(q_row), _ptr(s_row), layout,
                                 _stream(stream)), "mxfp4_quantize")


def mxfp4_quantize_dual(x, M, K, ldx, q_row, s_row, q_col, s_col, layout=MXFP4_SCALE_TC,
                        stream=None) -> None:
    _check(load().mxfp4_quantize_dual(_ptr(x), M, K, ldx, _ptr(q_row), _ptr(s_row), _ptr(q_col),
                                      _ptr(s_col), layout, _stream(stream)),
           "mxfp4_quantize_dual")


def mxfp4_quantize_dual_sr(x, M, K, ldx, q_row, s_row, q_col, s_col, layout=MXFP4_SCALE_TC,
                           seed=0, stream=None) -> None:
    _check(load().mxfp4_quantize_dual_sr(_ptr(x), M, K, ldx, _ptr(q_row), _ptr(s_row), _ptr(q_col),
                                         _ptr(s_col), layout, int(seed) & (2**64 - 1), _stream(stream)),
           "mxfp4_quantize_dual_sr")


def mxfp4_quantize_dual_2d(x, M, K, ldx, q_row, s_row, q_col, s_col, layout=MXFP4_SCALE_TC,
                           stream=None) -> None:
    _check(load().mxfp4_quantize_dual_2d(_ptr(x), M, K, ldx, _ptr(q_row), _ptr(s_row), _ptr(q_col),
                                         _ptr(s_col), layout, _stream(stream)),
           "mxfp4_quantize_dual_2d")


def mxfp4_quantize_dual_rht(x, M, K, ldx, q_row, s_row, q_col, s_col, layout=MXFP4_SCALE_TC,
                            signs=0, stream=None) -> None:
    _check(load().mxfp4_quantize_dual_rht(_ptr(x), M, K, ldx, _ptr(q_row), _ptr(s_row), _ptr(q_col),
                                          _ptr(s_col), layout, int(signs) & 0xFFFF, _stream(stream)),
           "mxfp4_quantize_dual_rht")


def mxfp4_quantize_dual_rht_sr(x, M, K, ldx, q_row, s_row, q_col, s_col, layout=MXFP4_SCALE_TC,
                               signs=0, seed=0, stream=None) -> None:
    _check(load().mxfp4_quantize_dual_rht_sr(_ptr(x), M, K, ldx, _ptr(q_row), _ptr(s_row), _ptr(q_col),
                                             _ptr(s_col), layout, int(signs) & 0xFFFF, int(seed) & (2**64 - 1),
                                             _stream(stream)),
           "mxfp4_quantize_dual_rht_sr")


def mxfp4_quantize_dual_qk_norm_rope_bwd(g, x, M, H, rstd, wq, wk, cos_table, sin_table, q_row, s_row, q_col,
                                         s_col, layout=MXFP4_SCALE_TC, dmixed=None, stream=None) -> None:
    _check(load().mxfp4_quantize_dual_qk_norm_rope_bwd(
        _ptr(g), _ptr(x), M, H, _ptr(rstd), _ptr(wq), _ptr(wk), _ptr(cos_table), _ptr(sin_table), _ptr(q_row),
        _ptr(s_row), _ptr(q_col), _ptr(s_col), layout, _ptr(dmixed), _stream(stream)),
        "mxfp4_quantize_dual_qk_norm_rope_bwd")


def quantize_qk_norm_rope_bwd(g, x, rstd, wq, wk, cos_table, sin_table, H, layout=MXFP4_SCALE_TC,
                              with_dmixed=False, stream=None):
    """Dual blobs of d(mixed_qkv) computed from the gradient g of the QK norm + RoPE output
    (bf16 [M, H*384], CUDA) in the quantizer's staging read: (row_q, row_s, col_q, col_s) and,
    with with_dmixed, the bf16 d(mixed_qkv) itself."""
    import torch
    M, K = g.shape
    assert K == 3 * H * 128 and x.shape == g.shape and g.dtype == x.dtype == torch.bfloat16
    rq, rs = alloc_blob(M, K, layout, g.device)
    cq, cs = alloc_blob(K, M, layout, g.device)
    dm = torch.empty_like(g) if with_dmixed else None
    mxfp4_quantize_dual_qk_norm_rope_bwd(g, x, M, H, rstd, wq, wk, cos_table, sin_table, rq, rs, cq, cs, layout, dm,
                                         stream)
    return (rq, rs, cq, cs, dm) if with_dmixed else (rq, rs, cq, cs)


def mxfp4_quantize_batch(tasks, dual: bool, layout=MXFP4_SCALE_TC, stream=None) -> None:
    """tasks: sequence of (x, rows, k, ldx, q_row, s_row, q_col, s_col[, flags[, rht_signs[,
    amax]]]); q_col / s_col may be None for the row-only quantizer; flags 0,
    MXFP4_QUANT_2D_BLOCKS or MXFP4_QUANT_RHT_COL; amax: None or a one-float CUDA buffer set
    to max |x| (the tensorwise FP8 amax)."""
    arr = (QuantizeTask * max(1, len(tasks)))()
    for i, t in enumerate(tasks):
        x, rows, k, ldx, q_row, s_row, q_col, s_col = t[:8]
        flags = t[8] if len(t) > 8 else 0
        signs = t[9] if len(t) > 9 else 0
        amax = t[10] if len(t) > 10 else None
        arr[i] = QuantizeTask(_ptr(x), rows, k, ldx, _ptr(q_row), _ptr(s_row), _ptr(q_col),
                              _ptr(s_col), flags, int(signs) & 0xFFFF, _ptr(amax))
    _check(load().mxfp4_quantize_batch(len(tasks), arr, int(bool(dual)), layout, _stream(stream)),
           "mxfp4_quantize_batch")


def mxfp4_gemm(a_q, a_s, b_q, b_s, M, N, K, c, ldc, out_dtype=MXFP4_OUT_BF16, stream=None) -> None:
    _check(load().mxfp4_gemm(_ptr(a_q), _ptr(a_s), _ptr(b_q), _ptr(b_s), M, N, K, _ptr(c), ldc,
                             out_dtype, _stream(stream)), "mxfp4_gemm")


def mxfp4_gemm_bias(a_q, a_s, b_q, b_s, M, N, K, bias, c, ldc, out_dtype=MXFP4_OUT_BF16,
                    stream=None) -> None:
    _check(load().mxfp4_gemm_bias(_ptr(a_q), _ptr(a_s), _ptr(b_q), _ptr(b_s), M, N, K, _ptr(bias),
                                  _ptr(c), ldc, out_dtype, _stream(stream)), "mxfp4_gemm_bias")


def mxfp4_gemm_quantize(a_q, a_s, b_q, b_s, M, N, K, bias, c, ldc, q_row, s_row, q_col=None, s_col=None,
                        stream=None) -> None:
    _check(load().mxfp4_gemm_quantize(_ptr(a_q), _ptr(a_s), _ptr(b_q), _ptr(b_s), M, N, K, _ptr(bias), _ptr(c),
                                      ldc, _ptr(q_row), _ptr(s_row), _ptr(q_col), _ptr(s_col), _stream(stream)),
           "mxfp4_gemm_quantize")


def gemm_quantize(a_q, a_s, b_q, b_s, M, N, K, dual=True, out=None, bias=None, stream=None):
    """bf16 C[M,N] = A . B^T (+ bias) and the MXFP4 blobs of C (tensor-core scale layout),
    as quantize(C, dual) would give them: (C, row_q, row_s[, col_q, col_s])."""
    import torch
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=a_q.device)
    assert out.dtype == torch.bfloat16 and out.stride(1) == 1
    rq, rs = alloc_blob(M, N, MXFP4_SCALE_TC, out.device)
    cq, cs = alloc_blob(N, M, MXFP4_SCALE_TC, out.device) if dual else (None, None)
    mxfp4_gemm_quantize(a_q, a_s, b_q, b_s, M, N, K, bias, out, out.stride(0), rq, rs, cq, cs, stream)
    return (out, rq, rs, cq, cs) if dual else (out, rq, rs)


def mxfp4_gemm_batch(tasks, stream=None) -> None:
    """tasks: sequence of (a_q, a_s, b_q, b_s, M, N, K, c, ldc, out_dtype[, bias])."""
    arr = (GemmTask * max(1, len(tasks)))()
    for i, t in enumerate(tasks):
        a_q, a_s, b_q, b_s, M, N, K, c, ldc, od = t[:10]
        bias = t[10] if len(t) > 10 else None
        arr[i] = GemmTask(_ptr(a_q), _ptr(a_s), _ptr(b_q), _ptr(b_s), M, N, K, _ptr(c), ldc, od, _ptr(bias))
    _check(load().mxfp4_gemm_batch(len(tasks), arr, _stream(stream)), "mxfp4_gemm_batch")


def mxfp4_gemm_set_tile_policy(policy) -> None:
    """MXFP4_TILES_AUTO / _NARROW / _WIDE for the CTA-pair GEMM launches that follow."""
    _check(load().mxfp4_gemm_set_tile_policy(policy), "mxfp4_gemm_set_tile_policy")


def mxfp4_fp8_quantize_tw(x, M, K, ldx, q_row, q_col, amax, scale_inv, stream=None) -> None:
    _check(load().mxfp4_fp8_quantize_tw(_ptr(x), M, K, ldx, _ptr(q_row), _ptr(q_col), _ptr(amax),
                                        _ptr(scale_inv), _stream(stream)), "mxfp4_fp8_quantize_tw")


def mxfp4_fp8_quantize_tw_batch(tasks, stream=None) -> None:
    """tasks: sequence of (x, M, K, ldx, q_row, q_col, amax, scale_inv[, amax_given]); q_row
    or q_col may be None; amax_given: amax already holds max |x| (from mxfp4_quantize_batch)."""
    arr = (Fp8QuantizeTask * max(1, len(tasks)))()
    for i, t in enumerate(tasks):
        x, M, K, ldx, qr, qc, amax, inv = t[:8]
        given = int(bool(t[8])) if len(t) > 8 else 0
        arr[i] = Fp8QuantizeTask(_ptr(x), M, K, ldx, _ptr(qr), _ptr(qc), _ptr(amax), _ptr(inv), given)
    _check(load().mxfp4_fp8_quantize_tw_batch(len(tasks), arr, _stream(stream)), "mxfp4_fp8_quantize_tw_batch")


def mxfp4_fp8_gemm(a, a_scale_inv, b, b_scale_inv, M, N, K, c, ldc, out_dtype=MXFP4_OUT_BF16,
                   stream=None) -> None:
    _check(load().mxfp4_fp8_gemm(_ptr(a), _ptr(a_scale_inv), _ptr(b), _ptr(b_scale_inv), M, N, K, _ptr(c),
                                 ldc, out_dtype, _stream(stream)), "mxfp4_fp8_gemm")


def mxfp4_fp8_gemm_batch(tasks, stream=None) -> None:
    """tasks: sequence of (a, a_scale_inv, b, b_scale_inv, M, N, K, c, ldc, out_dtype)."""
    arr = (Fp8GemmTask * max(1, len(tasks)))()
    for i, (a, sa, b, sb, M, N, K, c, ldc, od) in enumerate(tasks):
        arr[i] = Fp8GemmTask(_ptr(a), _ptr(sa), _ptr(b), _ptr(sb), M, N, K, _ptr(c), ldc, od)
    _check(load().mxfp4_fp8_gemm_batch(len(tasks), arr, _stream(stream)), "mxfp4_fp8_gemm_batch")


def _host_tasks(tasks):
    """tasks: sequence of (x, w, dy, y, dx, dw, M, N, K, train, out_dtype) with host
    buffers (tensors or addresses; dy, dx, dw may be None when train is 0)."""
    arr = (LinearHostTask * max(1, len(tasks)))()
    for i, (x, w, dy, y, dx, dw, M, N, K, train, od) in enumerate(tasks):
        arr[i] = LinearHostTask(_ptr(x), _ptr(w), _ptr(dy), _ptr(y), _ptr(dx), _ptr(dw), M, N, K,
                                int(bool(train)), od)
    return arr


def mxfp4_linear_workspace_bytes(tasks) -> int:
    n = ctypes.c_size_t()
    _check(load().mxfp4_linear_workspace_bytes(len(tasks), _host_tasks(tasks), ctypes.byref(n)),
           "mxfp4_linear_workspace_bytes")
    return n.value


def mxfp4_linear_step_host(tasks, workspace, workspace_bytes: int, stream=None) -> None:
    _check(load().mxfp4_linear_step_host(len(tasks), _host_tasks(tasks), _ptr(workspace),
                                         workspace_bytes, _stream(stream)), "mxfp4_linear_step_host")


def mxfp4_linear_pipelined_workspace_bytes(tasks) -> int:
    n = ctypes.c_size_t()
    _check(load().mxfp4_linear_pipelined_workspace_bytes(len(tasks), _host_tasks(tasks), ctypes.byref(n)),
           "mxfp4_linear_pipelined_workspace_bytes")
    return n.value


def mxfp4_linear_step_host_pipelined(tasks, workspace, workspace_bytes: int, stream=None) -> None:
    _check(load().mxfp4_linear_step_host_pipelined(len(tasks), _host_tasks(tasks), _ptr(workspace),
                                                   workspace_bytes, _stream(stream)),
           "mxfp4_linear_step_host_pipelined")


def mxfp4_linear_host_wait(stream=None) -> None:
    _check(load().mxfp4_linear_host_wait(_stream(stream)), "mxfp4_linear_host_wait")


def mxfp4_last_device_error(stream=None) -> int:
    """Returns the status (does not raise): MXFP4_ERR_TIMEOUT if a bounded wait ran out,
    MXFP4_ERR_NONFINITE if a tensorwise FP8 quantization met a non-finite input."""
    return int(load().mxfp4_last_device_error(_stream(stream)))


def mxfp4_selftest_bounded_wait(timeout_ns: int, stream=None) -> None:
    _check(load().mxfp4_selftest_bounded_wait(timeout_ns, _stream(stream)),
           "mxfp4_selftest_bounded_wait")


def mxfp4_status_string(status: int) -> str:
    return status_string(status)


# ---------------------------------------------------------------------------------------
# allocation helpers (torch as the allocator)
# ---------------------------------------------------------------------------------------
def alloc_blob(rows: int, k: int, layout: int = MXFP4_SCALE_TC, device="cuda"):
    """Uninitialised (q, s) uint8 buffers for one blob of `rows` rows and packed length k;
    q is shaped [rows, Kp/2], s is [rows, Kp/32] (plain) or flat (tensor-core layout)."""
    import torch
    qb, sb = mxfp4_quantize_sizes(rows, k, layout)
    kp = (k + 127) // 128 * 128
    q = torch.empty((rows, kp // 2), dtype=torch.uint8, device=device)
    if layout == MXFP4_SCALE_PLAIN:
        s = torch.empty((rows, kp // 32), dtype=torch.uint8, device=device)
    else:
        s = torch.empty((sb,), dtype=torch.uint8, device=device)
    assert q.numel() == qb and s.numel() == sb
    return q, s


def quantize(x, dual: bool = True, layout: int = MXFP4_SCALE_TC, stream=None, sr_seed=None,
             block_2d: bool = False, rht_signs=None):
    """bf16 X[M,K] (CUDA, row pitch a multiple of 8) -> (row_q, row_s[, col_q, col_s]);
    with sr_seed (dual only) the elements are stochastically rounded; with block_2d the
    scales are those of 32 x 32 blocks; with rht_signs (dual only) the col blob is that of
    the Hadamard-transformed columns (both: the gradient recipe with stochastic rounding)."""
    import torch
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    M, K = x.shape
    rq, rs = alloc_blob(M, K, layout, x.device)
    if rht_signs is not None:
        assert dual and not block_2d
        cq, cs = alloc_blob(K, M, layout, x.device)
        if sr_seed is None:
            mxfp4_quantize_dual_rht(x, M, K, x.stride(0), rq, rs, cq, cs, layout, rht_signs, stream)
        else:
            mxfp4_quantize_dual_rht_sr(x, M, K, x.stride(0), rq, rs, cq, cs, layout, rht_signs, sr_seed, stream)
        return rq, rs, cq, cs
    if block_2d:
        assert sr_seed is None, "the 2-D block recipe is for weights, stochastic rounding for gradients"
        if not dual:
            mxfp4_quantize_batch([(x, M, K, x.stride(0), rq, rs, None, None, MXFP4_QUANT_2D_BLOCKS)], False,
                                 layout, stream)
            return rq, rs
        cq, cs = alloc_blob(K, M, layout, x.device)
        mxfp4_quantize_dual_2d(x, M, K, x.stride(0), rq, rs, cq, cs, layout, stream)
        return rq, rs, cq, cs
    if not dual:
        assert sr_seed is None, "stochastic rounding is a mode of the dual quantizer"
        mxfp4_quantize(x, M, K, x.stride(0), rq, rs, layout, stream)
        return rq, rs
    cq, cs = alloc_blob(K, M, layout, x.device)
    if sr_seed is None:
        mxfp4_quantize_dual(x, M, K, x.stride(0), rq, rs, cq, cs, layout, stream)
    else:
        mxfp4_quantize_dual_sr(x, M, K, x.stride(0), rq, rs, cq, cs, layout, sr_seed, stream)
    return rq, rs, cq, cs


def gemm(a_q, a_s, b_q, b_s, M, N, K, out_dtype=None, out=None, stream=None, bias=None):
    """C[M,N] = A . B^T (+ bias[N], a contiguous bf16 vector, when given) from two K-packed
    blobs with tensor-core-layout scales."""
    import torch
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype or torch.bfloat16, device=a_q.device)
    code = MXFP4_OUT_F32 if out.dtype == torch.float32 else MXFP4_OUT_BF16
    assert out.dtype in (torch.float32, torch.bfloat16) and out.stride(1) == 1
    if bias is None:
        mxfp4_gemm(a_q, a_s, b_q, b_s, M, N, K, out, out.stride(0), code, stream)
    else:
        assert bias.dtype == torch.bfloat16 and bias.is_contiguous() and bias.numel() == N
        mxfp4_gemm_bias(a_q, a_s, b_q, b_s, M, N, K, bias, out, out.stride(0), code, stream)
    return out


def fp8_pitch(n: int) -> int:
    """Row pitch in bytes of an E5M2 copy whose rows hold n elements (16-byte rounded)."""
    return (n + 15) // 16 * 16


def fp8_quantize(x, row: bool = True, col: bool = True, scalars=None, stream=None):
    """Tensorwise E5M2 quantization of bf16 X[M,K] (CUDA): (q_row [M, pitch(K)] or None,
    q_col [K, pitch(M)] or None, amax, scale_inv), the last two one-element fp32 CUDA
    tensors (views into `scalars`, a 2-element fp32 tensor, when given)."""
    import torch
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    M, K = x.shape
    qr = torch.empty((M, fp8_pitch(K)), dtype=torch.uint8, device=x.device) if row else None
    qc = torch.empty((K, fp8_pitch(M)), dtype=torch.uint8, device=x.device) if col else None
    if scalars is None:
        scalars = torch.empty(2, dtype=torch.float32, device=x.device)
    amax, inv = scalars[0:1], scalars[1:2]
    mxfp4_fp8_quantize_tw(x, M, K, x.stride(0), qr, qc, amax, inv, stream)
    return qr, qc, amax, inv


def fp8_gemm(a, a_scale_inv, b, b_scale_inv, M, N, K, out_dtype=None, out=None, stream=None):
    """C[M,N] = (A . B^T) * a_scale_inv * b_scale_inv over E5M2 codes A [M, pitch(K)],
    B [N, pitch(K)]."""
    import torch
    if out is None:
        out = torch.empty((M, N), dtype=out_dtype or torch.bfloat16, device=a.device)
    code = MXFP4_OUT_F32 if out.dtype == torch.float32 else MXFP4_OUT_BF16
    assert out.dtype in (torch.float32, torch.bfloat16) and out.stride(1) == 1
    mxfp4_fp8_gemm(a, a_scale_inv, b, b_scale_inv, M, N, K, out, out.stride(0), code, stream)
    return out
