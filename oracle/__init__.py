"""CPU oracle for MXFP4 block-scaled quantization and GEMM (numpy front end over the C
code in mxfp4_oracle.c).

TEST INFRASTRUCTURE ONLY: imported by the tests, by the package's smoke check and by
the benchmark's CPU-baseline leg, never by the product path.  It shares no code with the
CUDA library.  The arithmetic and the passages it follows are documented in
mxfp4_oracle.c; this module only marshals numpy arrays.

Parity status: every function here is pinned by the oracle self-tests
(tests/test_oracle_*.py; the bias add against torch's own CPU elementwise add, the
operation the layer performs) except the tensor-core scale layout, whose byte positions are a
layout of this library's own choosing; that permutation is pinned on the CPU only as a
bijection, and against the hardware by the GEMM parity tests.
"""
import ctypes
import numpy as np

from . import build as _build

BLOCK = 32   # MXFP4_BLOCK_SIZE
PAD = 128    # MXFP4_PADDING_ALIGN_SIZE

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        i64, u8, u16, f64 = ctypes.c_int64, ctypes.c_uint8, ctypes.c_uint16, ctypes.c_double
        vp = ctypes.c_void_p
        lib.oracle_bf16_to_f64.argtypes = [u16]
        lib.oracle_bf16_to_f64.restype = f64
        lib.oracle_e2m1_decode.argtypes = [u8]
        lib.oracle_e2m1_decode.restype = f64
        lib.oracle_e2m1_encode.argtypes = [f64]
        lib.oracle_e2m1_encode.restype = u8
        lib.oracle_e8m0_scale.argtypes = [f64]
        lib.oracle_e8m0_scale.restype = u8
        for fn in (lib.oracle_quantize_row, lib.oracle_quantize_col):
            fn.argtypes = [vp, i64, i64, i64, vp, vp]
            fn.restype = ctypes.c_int
        lib.oracle_scale_to_tc.argtypes = [vp, i64, i64, vp]
        lib.oracle_scale_to_tc.restype = None
        lib.oracle_dequantize.argtypes = [vp, vp, i64, i64, vp]
        lib.oracle_dequantize.restype = None
        lib.oracle_gemm_f64.argtypes = [vp, vp, i64, i64, i64, i64, i64, vp, vp]
        lib.oracle_gemm_f64.restype = None
        lib.oracle_round_to_bf16.argtypes = [vp, vp, i64]
        lib.oracle_round_to_bf16.restype = None
        for fn in (lib.oracle_bias_add_bf16, lib.oracle_bias_add_f32):
            fn.argtypes = [vp, vp, i64, i64, vp]
            fn.restype = None
        for fn in (lib.oracle_quantize_row_2d, lib.oracle_quantize_col_2d):
            fn.argtypes = [vp, i64, i64, i64, vp, vp]
            fn.restype = ctypes.c_int
        lib.oracle_e5m2_decode.argtypes = [u8]
        lib.oracle_e5m2_decode.restype = f64
        lib.oracle_e5m2_encode.argtypes = [f64]
        lib.oracle_e5m2_encode.restype = u8
        lib.oracle_fp8_quantize_tw.argtypes = [vp, i64, i64, i64, vp, i64, vp, i64, vp, vp]
        lib.oracle_fp8_quantize_tw.restype = ctypes.c_int
        lib.oracle_fp8_dequantize.argtypes = [vp, i64, i64, i64, vp]
        lib.oracle_fp8_dequantize.restype = None
        lib.oracle_fp8_output_scale.argtypes = [ctypes.c_float, ctypes.c_float]
        lib.oracle_fp8_output_scale.restype = ctypes.c_float
        lib.oracle_philox4x32_10.argtypes = [vp, vp, vp]
        lib.oracle_philox4x32_10.restype = None
        lib.oracle_sr_bits.argtypes = [ctypes.c_uint64, i64, i64, ctypes.c_int]
        lib.oracle_sr_bits.restype = ctypes.c_uint32
        lib.oracle_e2m1_encode_sr.argtypes = [f64, ctypes.c_uint32]
        lib.oracle_e2m1_encode_sr.restype = u8
        for fn in (lib.oracle_quantize_row_sr, lib.oracle_quantize_col_sr):
            fn.argtypes = [vp, i64, i64, i64, vp, vp, ctypes.c_uint64, vp]
            fn.restype = ctypes.c_int
        lib.oracle_rht16.argtypes = [vp, ctypes.c_uint32]
        lib.oracle_rht16.restype = None
        lib.oracle_quantize_col_rht.argtypes = [vp, i64, i64, i64, ctypes.c_uint32, vp, vp]
        lib.oracle_quantize_col_rht.restype = ctypes.c_int
        lib.oracle_quantize_col_rht_sr.argtypes = [vp, i64, i64, i64, ctypes.c_uint32, vp, vp, ctypes.c_uint64, vp]
        lib.oracle_quantize_col_rht_sr.restype = ctypes.c_int
        lib.oracle_qk_norm_rope_fwd.argtypes = [vp, vp, vp, vp, vp, f64, i64, i64, i64, vp, vp]
        lib.oracle_qk_norm_rope_fwd.restype = None
        lib.oracle_qk_norm_rope_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, vp]
        lib.oracle_qk_norm_rope_bwd.restype = None
        _lib = lib
    return _lib


def cdiv(a, b):
    return (a + b - 1) // b


def padded(n):
    """Length of the packed dimension after padding to MXFP4_PADDING_ALIGN_SIZE."""
    return cdiv(n, PAD) * PAD


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _bits(x):
    x = np.asarray(x)
    if x.dtype != np.uint16:
        raise TypeError("oracle inputs are bf16 bit patterns (numpy uint16)")
    return np.ascontiguousarray(x)


# ---- scalar codecs -------------------------------------------------------------------
def bf16_to_f64(bits):
    return _load().oracle_bf16_to_f64(int(bits))


def e2m1_decode(code):
    return _load().oracle_e2m1_decode(int(code))


def e2m1_encode(v):
    return int(_load().oracle_e2m1_encode(float(v)))


def e8m0_scale(amax):
    return int(_load().oracle_e8m0_scale(float(amax)))


# ---- quantizers ------------------------------------------------------------------------
def quantize_row(x_bits):
    """Row blob of X[M,K]: (q[M, Kp/2] u8, s[M, Kp/32] u8, plain scale layout)."""
    x = _bits(x_bits)
    M, K = x.shape
    Kp = padded(K)
    q = np.zeros((M, Kp // 2), np.uint8)
    s = np.zeros((M, Kp // BLOCK), np.uint8)
    if M and K and _load().oracle_quantize_row(_ptr(x), M, K, K, _ptr(q), _ptr(s)):
        raise ValueError("oracle: non-finite input")
    return q, s


def quantize_col(x_bits):
    """Col blob of X[M,K] = row blob of X^T: (q[K, Mp/2] u8, s[K, Mp/32] u8)."""
    x = _bits(x_bits)
    M, K = x.shape
    Mp = padded(M)
    q = np.zeros((K, Mp // 2), np.uint8)
    s = np.zeros((K, Mp // BLOCK), np.uint8)
    if M and K and _load().oracle_quantize_col(_ptr(x), M, K, K, _ptr(q), _ptr(s)):
        raise ValueError("oracle: non-finite input")
    return q, s


def quantize_dual(x_bits):
    """(row_q, row_s, col_q, col_s), the four outputs of the dual quantizer."""
    rq, rs = quantize_row(x_bits)
    cq, cs = quantize_col(x_bits)
    return rq, rs, cq, cs


def scale_to_tc(s_plain):
    """Plain scale bytes [R, KB] -> tensor-core layout, flat u8 of ceil(R/128)*128*KB."""
    s = np.ascontiguousarray(s_plain, dtype=np.uint8)
    R, KB = s.shape
    out = np.empty(padded(R) * KB, np.uint8)
    _load().oracle_scale_to_tc(_ptr(s), R, KB, _ptr(out))
    return out


# ---- GEMM -------------------------------------------------------------------------------
def dequantize(q, s):
    """Blob (q[R, Kp/2], plain s[R, Kp/32]) -> fp64 [R, Kp]."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    s = np.ascontiguousarray(s, dtype=np.uint8)
    R, half = q.shape
    Kp = half * 2
    assert s.shape == (R, Kp // BLOCK)
    out = np.empty((R, Kp), np.float64)
    _load().oracle_dequantize(_ptr(q), _ptr(s), R, Kp, _ptr(out))
    return out


def gemm_dequantized(a, b, rows=None, want_abs=True):
    """C = A . B^T over fp64 dequantized operands A[M,Kp], B[N,Kp] (rows of C limited to
    the range `rows` = (m0, m1) when given).  Returns (C, sum_k |a_k b_k|)."""
    a = np.ascontiguousarray(a, dtype=np.float64)
    b = np.ascontiguousarray(b, dtype=np.float64)
    M, Kp = a.shape
    N, Kb = b.shape
    assert Kb == Kp
    m0, m1 = rows if rows is not None else (0, M)
    c = np.empty((m1 - m0, N), np.float64)
    cabs = np.empty((m1 - m0, N), np.float64) if want_abs else None
    _load().oracle_gemm_f64(_ptr(a), _ptr(b), M, N, Kp, m0, m1, _ptr(c),
                            _ptr(cabs) if want_abs else None)
    return c, cabs


def gemm(aq, a_s, bq, b_s, rows=None, want_abs=True):
    """C[M,N] = A . B^T from two K-packed blobs in the plain scale layout."""
    return gemm_dequantized(dequantize(aq, a_s), dequantize(bq, b_s), rows, want_abs)


def round_to_bf16(x):
    """fp64 -> bf16 bit patterns, one round-to-nearest-even."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, np.uint16)
    _load().oracle_round_to_bf16(_ptr(x), _ptr(out), x.size)
    return out


def round_to_f32(x):
    """fp64 -> binary32, one round-to-nearest-even (numpy's cast)."""
    return np.asarray(x, dtype=np.float64).astype(np.float32)


def bias_add(y, bias_bits):
    """The layer's `output + bias` after the GEMM: y is the GEMM output already in its
    dtype (bf16 bit patterns as uint16 [M, N], or float32 [M, N]), bias_bits the bf16 bias
    [N] as uint16.  Returns the same dtype as y."""
    bias_bits = np.ascontiguousarray(bias_bits, dtype=np.uint16)
    if y.dtype == np.uint16:
        y = np.ascontiguousarray(y)
        M, N = y.shape
        assert bias_bits.shape == (N,)
        out = np.empty((M, N), np.uint16)
        _load().oracle_bias_add_bf16(_ptr(y), _ptr(bias_bits), M, N, _ptr(out))
        return out
    y = np.ascontiguousarray(y, dtype=np.float32)
    M, N = y.shape
    assert bias_bits.shape == (N,)
    out = np.empty((M, N), np.float32)
    _load().oracle_bias_add_f32(_ptr(y), _ptr(bias_bits), M, N, _ptr(out))
    return out


# --- stochastic rounding (the gradient quantizer's `use_sr` flag) -------------------------

def philox4x32_10(ctr, key):
    """Philox4x32-10 of a 4-word counter and a 2-word key -> 4 words (uint32)."""
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.empty(4, np.uint32)
    _load().oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def sr_bits(seed, a, b, packing):
    """16 random bits of element (row a, column b) of the row (0) or col (1) blob."""
    return int(_load().oracle_sr_bits(int(seed) & (2**64 - 1), int(a), int(b), int(packing)))


def e2m1_encode_sr(y, r):
    """E2M1 code of the scaled element y with stochastic rounding driven by 16 bits r."""
    return int(_load().oracle_e2m1_encode_sr(float(y), int(r)))


def _ids(ids, n):
    if ids is None:
        return None
    ids = np.ascontiguousarray(ids, dtype=np.int64)
    assert ids.shape == (n,)
    return ids


def quantize_row_sr(x_bits, seed, row_ids=None):
    """Row blob of X[M,K] with stochastically rounded elements (plain scale layout);
    row_ids: each row's index in the full tensor when x_bits holds sampled rows."""
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    M, K = x_bits.shape
    Kp = padded(K)
    q = np.empty((M, Kp // 2), np.uint8)
    s = np.empty((M, Kp // BLOCK), np.uint8)
    ids = _ids(row_ids, M)
    if _load().oracle_quantize_row_sr(_ptr(x_bits), M, K, K, _ptr(q), _ptr(s), int(seed) & (2**64 - 1),
                                      None if ids is None else _ptr(ids)):
        raise ValueError("non-finite input")
    return q, s


def quantize_col_sr(x_bits, seed, col_ids=None):
    """Col blob of X[M,K] (row blob of X^T) with stochastically rounded elements;
    col_ids: each column's index in the full tensor when x_bits holds sampled columns."""
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    M, K = x_bits.shape
    Mp = padded(M)
    q = np.empty((K, Mp // 2), np.uint8)
    s = np.empty((K, Mp // BLOCK), np.uint8)
    ids = _ids(col_ids, K)
    if _load().oracle_quantize_col_sr(_ptr(x_bits), M, K, K, _ptr(q), _ptr(s), int(seed) & (2**64 - 1),
                                      None if ids is None else _ptr(ids)):
        raise ValueError("non-finite input")
    return q, s


def quantize_dual_sr(x_bits, seed):
    """(row_q, row_s, col_q, col_s) of the dual quantizer with stochastic rounding."""
    return quantize_row_sr(x_bits, seed) + quantize_col_sr(x_bits, seed)


# --- hybrid FP8 backward: tensorwise E5M2 quantization and the FP8 GEMM ---------------

FP8_PITCH = 16   # row pitch of the E5M2 copies: a multiple of 16 bytes


def fp8_pitch(n):
    """Row pitch in bytes of an E5M2 copy whose rows hold n elements."""
    return cdiv(n, FP8_PITCH) * FP8_PITCH


def e5m2_decode(code):
    return float(_load().oracle_e5m2_decode(int(code)))


def e5m2_encode(v):
    return int(_load().oracle_e5m2_encode(float(v)))


def fp8_quantize_tw(x_bits, row=True, col=True):
    """Tensorwise E5M2 quantization of X[M,K] (bf16 bits): (q_row [M, pitch(K)] or None,
    q_col [K, pitch(M)] or None, amax, scale_inv), padding bytes 0x00."""
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    M, K = x_bits.shape
    qr = np.empty((M, fp8_pitch(K)), np.uint8) if row else None
    qc = np.empty((K, fp8_pitch(M)), np.uint8) if col else None
    amax = np.zeros(1, np.float32)
    inv = np.zeros(1, np.float32)
    if _load().oracle_fp8_quantize_tw(_ptr(x_bits), M, K, K, None if qr is None else _ptr(qr), fp8_pitch(K),
                                      None if qc is None else _ptr(qc), fp8_pitch(M), _ptr(amax), _ptr(inv)):
        raise ValueError("non-finite input")
    return qr, qc, float(amax[0]), float(inv[0])


def fp8_dequantize(q, cols):
    """E5M2 codes [R, pitch] -> fp64 [R, cols]."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    R, ld = q.shape
    out = np.empty((R, cols), np.float64)
    _load().oracle_fp8_dequantize(_ptr(q), R, cols, ld, _ptr(out))
    return out


def fp8_output_scale(a_scale_inv, b_scale_inv):
    return float(_load().oracle_fp8_output_scale(a_scale_inv, b_scale_inv))


def fp8_gemm(a_q, a_scale_inv, b_q, b_scale_inv, K, rows=None):
    """C = (A . B^T) * s over E5M2 codes A [M, pitch], B [N, pitch] (first K columns), s the
    binary32 product of the inverse scales; returns (C, sum_k |a_k b_k| * s) in fp64."""
    a = fp8_dequantize(a_q if rows is None else np.ascontiguousarray(a_q[rows]), K)
    b = fp8_dequantize(b_q, K)
    c, cabs = gemm_dequantized(a, b)
    s = fp8_output_scale(a_scale_inv, b_scale_inv)
    return c * s, cabs * s


# --- 2-D (32 x 32) block scales for weights ---------------------------------------------

def quantize_row_2d(x_bits):
    """Row blob of X[M,K] with one scale per 32 x 32 block (plain scale layout)."""
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    M, K = x_bits.shape
    Kp = padded(K)
    q = np.empty((M, Kp // 2), np.uint8)
    s = np.empty((M, Kp // BLOCK), np.uint8)
    if _load().oracle_quantize_row_2d(_ptr(x_bits), M, K, K, _ptr(q), _ptr(s)):
        raise ValueError("non-finite input")
    return q, s


def quantize_col_2d(x_bits):
    """Col blob of X[M,K] with the same 32 x 32 block scales."""
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    M, K = x_bits.shape
    Mp = padded(M)
    q = np.empty((K, Mp // 2), np.uint8)
    s = np.empty((K, Mp // BLOCK), np.uint8)
    if _load().oracle_quantize_col_2d(_ptr(x_bits), M, K, K, _ptr(q), _ptr(s)):
        raise ValueError("non-finite input")
    return q, s


# --- Hadamard transform of the column blobs (`colwise_use_rht`) -------------------------

def rht16(v, signs):
    """The 16-point transform (1/4) H16 diag(s) of 16 values, in fp32 (returns float32)."""
    a = np.ascontiguousarray(np.asarray(v, dtype=np.float32).reshape(16)).copy()
    _load().oracle_rht16(_ptr(a), int(signs) & 0xFFFF)
    return a


def quantize_col_rht(x_bits, signs):
    """Col blob of X[M,K] with the 16-point transform applied along M (plain scale layout)."""
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    M, K = x_bits.shape
    Mp = padded(M)
    q = np.empty((K, Mp // 2), np.uint8)
    s = np.empty((K, Mp // BLOCK), np.uint8)
    if _load().oracle_quantize_col_rht(_ptr(x_bits), M, K, K, int(signs) & 0xFFFF, _ptr(q), _ptr(s)):
        raise ValueError("non-finite input or transform")
    return q, s


def quantize_col_rht_sr(x_bits, signs, seed, col_ids=None):
    """Col blob of X[M,K] with the 16-point transform applied along M and stochastically
    rounded elements (the gradient recipe with `use_sr`); col_ids: each column's index in
    the full tensor when x_bits holds sampled columns."""
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    M, K = x_bits.shape
    Mp = padded(M)
    q = np.empty((K, Mp // 2), np.uint8)
    s = np.empty((K, Mp // BLOCK), np.uint8)
    ids = _ids(col_ids, K)
    if _load().oracle_quantize_col_rht_sr(_ptr(x_bits), M, K, K, int(signs) & 0xFFFF, _ptr(q), _ptr(s),
                                          int(seed) & (2**64 - 1), None if ids is None else _ptr(ids)):
        raise ValueError("non-finite input or transform")
    return q, s


# --- QK RMSNorm + interleaved RoPE backward (the quantizer prologue) -----------------------

def qk_norm_rope_fwd(mixed, wq, wk, cos, sin, H, D, eps=1e-6):
    """Forward of the norm + RoPE over fp64 mixed[M, H*3*D]: (out [M, H*3*D] with v copied,
    r [M, H, 2] the saved 1/sqrt(mean(x^2) + eps) of q and k)."""
    mixed = np.ascontiguousarray(mixed, dtype=np.float64)
    M = mixed.shape[0]
    assert mixed.shape[1] == 3 * H * D
    c = [np.ascontiguousarray(a, dtype=np.float64) for a in (wq, wk, cos, sin)]
    out = np.empty_like(mixed)
    r = np.empty((M, H, 2), np.float64)
    _load().oracle_qk_norm_rope_fwd(_ptr(mixed), *(_ptr(a) for a in c), float(eps), M, H, D, _ptr(out), _ptr(r))
    return out, r


def qk_norm_rope_bwd(g_bits, x_bits, r, wq, wk, cos, sin, H, D):
    """d(mixed_qkv) [M, H*3*D] in fp64 from bf16 g (the gradient of the norm + RoPE output,
    v part: the gradient of v) and x (mixed_qkv), the saved r [M, H, 2] and the fp32 norm
    weights and RoPE tables."""
    g_bits = np.ascontiguousarray(g_bits, dtype=np.uint16)
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    M = g_bits.shape[0]
    assert g_bits.shape == x_bits.shape == (M, 3 * H * D)
    f = [np.ascontiguousarray(a, dtype=np.float32) for a in (r, wq, wk, cos, sin)]
    out = np.empty((M, 3 * H * D), np.float64)
    _load().oracle_qk_norm_rope_bwd(_ptr(g_bits), _ptr(x_bits), *(_ptr(a) for a in f), M, H, D, _ptr(out))
    return out

