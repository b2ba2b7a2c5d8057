"""Shared comparison helpers for the GPU parity tests (test infrastructure).

The comparisons follow the accuracy contract of the library:
  - quantized bytes and scale bytes: bit-exact against the oracle, padding included;
  - fp32 GEMM output: |gpu - oracle| <= 1e-5 * sum_k |a_k b_k| per element;
  - bf16 GEMM output: within 1 bf16 ulp of the oracle's fp64 result rounded once to bf16,
    or, for outputs that nearly cancel (where the fp32 accumulation the hardware performs
    is itself allowed 1e-5 * sum_k |a_k b_k|), within that bound plus one bf16 ulp.
"""
import json
import os

import numpy as np
import torch

import oracle
from mxfp4_block_scaled_quantize_gb300 import abi, workloads

FP32_REL = 1e-5
# At most this fraction of a bf16 GEMM's outputs may pass only through the near-cancel
# clause (more than 1 ulp from the rounded oracle, within 1e-5 * sum|ab| + 1 ulp of it):
# those are outputs whose sum cancels so deeply that the fp32 accumulation error reaches
# half a bf16 ulp of the result, which random inputs make rare.
MAX_NEAR_CANCEL_FRAC = 0.01


def log_stats(what: str, stats: dict) -> None:
    """Appends one JSON line of comparison statistics to $MXFP4_PARITY_LOG, when set."""
    path = os.environ.get("MXFP4_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"what": what, **stats}) + "\n")


def to_gpu(x_cpu: torch.Tensor, device="cuda:0") -> torch.Tensor:
    return x_cpu.to(device)


def tc_index(r, kb, KB):
    """Flat position of scale byte (r, kb) in the tensor-core layout (test-side helper)."""
    r = np.asarray(r, np.int64)
    kb = np.asarray(kb, np.int64)
    return ((r // 128) * (KB // 4) + kb // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + kb % 4


def gather_tc_rows(s_tc: np.ndarray, rows: np.ndarray, KB: int) -> np.ndarray:
    rr, kk = np.meshgrid(rows, np.arange(KB), indexing="ij")
    return s_tc[tc_index(rr, kk, KB)]


def assert_bytes_equal(got: np.ndarray, want: np.ndarray, what: str) -> None:
    got = np.asarray(got)
    want = np.asarray(want)
    assert got.shape == want.shape, f"{what}: shape {got.shape} != {want.shape}"
    bad = np.nonzero(got != want)
    if bad[0].size:
        idx = tuple(b[0] for b in bad)
        raise AssertionError(f"{what}: {bad[0].size} bytes differ; first at {idx}: "
                             f"gpu {got[idx]:#04x} oracle {want[idx]:#04x}")


def check_quantized_full(x_cpu: torch.Tensor, outs, layout: int, dual: bool, what: str) -> None:
    """Every byte of the GPU blobs (row, and col when dual) equals the oracle's."""
    xb = workloads.bf16_bits(x_cpu)
    M, K = xb.shape
    rq, rs = oracle.quantize_row(xb)
    assert_bytes_equal(outs[0].cpu().numpy(), rq, f"{what} row q")
    srs = rs if layout == abi.MXFP4_SCALE_PLAIN else oracle.scale_to_tc(rs)
    assert_bytes_equal(outs[1].cpu().numpy().reshape(srs.shape), srs, f"{what} row s")
    if dual:
        cq, cs = oracle.quantize_col(xb)
        assert_bytes_equal(outs[2].cpu().numpy(), cq, f"{what} col q")
        scs = cs if layout == abi.MXFP4_SCALE_PLAIN else oracle.scale_to_tc(cs)
        assert_bytes_equal(outs[3].cpu().numpy().reshape(scs.shape), scs, f"{what} col s")


def check_quantized_sampled(x_cpu: torch.Tensor, outs, dual: bool, what: str, n_rows=48,
                            n_cols=48, seed=0) -> None:
    """Large inputs: the oracle quantizes sampled rows (row blob) and sampled columns (col
    blob: whole columns, so every column block is complete) and they must match the GPU's
    bytes at those rows; scales are read from the tensor-core layout."""
    xb = workloads.bf16_bits(x_cpu)
    M, K = xb.shape
    rng = np.random.default_rng(seed)
    rows = np.unique(np.concatenate([rng.choice(M, min(n_rows, M), replace=False),
                                     [0, M - 1, min(M - 1, 127), min(M - 1, 128)]]))
    rq, rs = oracle.quantize_row(np.ascontiguousarray(xb[rows]))
    g_rq = outs[0][torch.as_tensor(rows, device=outs[0].device)].cpu().numpy()
    assert_bytes_equal(g_rq, rq, f"{what} row q (sampled)")
    KB = rs.shape[1]
    assert_bytes_equal(gather_tc_rows(outs[1].cpu().numpy(), rows, KB), rs, f"{what} row s (sampled)")
    if dual:
        cols = np.unique(np.concatenate([rng.choice(K, min(n_cols, K), replace=False),
                                         [0, K - 1]]))
        cq, cs = oracle.quantize_col(np.ascontiguousarray(xb[:, cols]))
        g_cq = outs[2][torch.as_tensor(cols, device=outs[2].device)].cpu().numpy()
        assert_bytes_equal(g_cq, cq, f"{what} col q (sampled)")
        MB = cs.shape[1]
        assert_bytes_equal(gather_tc_rows(outs[3].cpu().numpy(), cols, MB), cs,
                           f"{what} col s (sampled)")


def check_rows_cols(x_cpu: torch.Tensor, outs, rows, cols, what: str) -> None:
    """The row blob at the given rows and the col blob at the given columns of X equal the
    oracle's (scales read from the tensor-core layout)."""
    xb = workloads.bf16_bits(x_cpu)
    rows = np.unique(np.asarray(rows))
    cols = np.unique(np.asarray(cols))
    rq, rs = oracle.quantize_row(np.ascontiguousarray(xb[rows]))
    assert_bytes_equal(outs[0][torch.as_tensor(rows, device=outs[0].device)].cpu().numpy(), rq, f"{what} row q")
    assert_bytes_equal(gather_tc_rows(outs[1].cpu().numpy(), rows, rs.shape[1]), rs, f"{what} row s")
    cq, cs = oracle.quantize_col(np.ascontiguousarray(xb[:, cols]))
    assert_bytes_equal(outs[2][torch.as_tensor(cols, device=outs[2].device)].cpu().numpy(), cq, f"{what} col q")
    assert_bytes_equal(gather_tc_rows(outs[3].cpu().numpy(), cols, cs.shape[1]), cs, f"{what} col s")


def tc_to_plain(s_tc: np.ndarray, R: int, KB: int) -> np.ndarray:
    return gather_tc_rows(s_tc, np.arange(R), KB)


def bf16_key(bits: np.ndarray) -> np.ndarray:
    b = bits.astype(np.int64)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def bf16_ulp(ref: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |ref| (subnormal spacing 2^-133 at the bottom)."""
    a = np.abs(ref)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -126)
    return np.ldexp(1.0, (e - 7).astype(np.int64))


def check_gemm(c_gpu: torch.Tensor, c_ref: np.ndarray, cabs: np.ndarray, what: str) -> dict:
    """c_gpu: rows of the GPU output matching c_ref (fp64 oracle) and cabs."""
    if c_gpu.dtype == torch.float32:
        g = c_gpu.cpu().numpy().astype(np.float64)
        err = np.abs(g - c_ref)
        bound = FP32_REL * cabs
        bad = err > bound
        if bad.any():
            i = np.argwhere(bad)[0]
            raise AssertionError(f"{what}: {bad.sum()} fp32 outputs out of bound; first {tuple(i)}: "
                                 f"gpu {g[tuple(i)]!r} oracle {c_ref[tuple(i)]!r} bound {bound[tuple(i)]!r}")
        stats = {"n": int(err.size), "max_err_over_bound": float(np.max(err / np.maximum(bound, 1e-300)))}
        log_stats(what, stats)
        return stats
    assert c_gpu.dtype == torch.bfloat16
    gbits = c_gpu.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    rbits = oracle.round_to_bf16(c_ref)
    ulps = np.abs(bf16_key(gbits) - bf16_key(rbits))
    g = (gbits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    near_cancel_ok = np.abs(g - c_ref) <= FP32_REL * cabs + bf16_ulp(c_ref)
    bad = (ulps > 1) & ~near_cancel_ok
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {bad.sum()} bf16 outputs off by more than 1 ulp; first {i}: "
                             f"gpu {g[i]!r} oracle {c_ref[i]!r} ({ulps[i]} ulp)")
    stats = {"within_1ulp": int(np.sum(ulps <= 1)), "near_cancel": int(np.sum(ulps > 1)),
             "exact": int(np.sum(ulps == 0)), "n": int(ulps.size)}
    log_stats(what, stats)
    # (a fraction says nothing about a handful of outputs: applied from 1000 outputs up)
    assert stats["n"] < 1000 or stats["near_cancel"] <= MAX_NEAR_CANCEL_FRAC * stats["n"], (
        f"{what}: {stats['near_cancel']} of {stats['n']} bf16 outputs pass only as near-cancelling sums")
    return stats


def oracle_gemm_rows(a_q, a_s_plain, b_q, b_s_plain, rows):
    """fp64 oracle for the given output rows only: (C[rows], sum|ab|[rows])."""
    a = oracle.dequantize(a_q[rows], a_s_plain[rows])
    b = oracle.dequantize(b_q, b_s_plain)
    return oracle.gemm_dequantized(a, b)


def _bf16_from_key(k: np.ndarray) -> np.ndarray:
    k = np.asarray(k, np.int64)
    return np.where(k >= 0, k, 0x8000 | (-k)).astype(np.uint16)


def check_gemm_bias(c_gpu: torch.Tensor, c_ref: np.ndarray, cabs: np.ndarray, bias_bits: np.ndarray,
                    what: str) -> dict:
    """GEMM output with the fused bias add (the layer's `output + bias`).  The oracle applies
    its bias add to its own GEMM result in the output dtype:
      - fp32: |gpu - oracle| <= 1e-5 * sum|ab| + one fp32 spacing at the result;
      - bf16: the GPU value is the oracle's bias add of the oracle's bf16 GEMM output or of
        one of its two bf16 neighbours (the GEMM is allowed 1 ulp), or, where the GEMM
        nearly cancels, within 1e-5 * sum|ab| plus two bf16 ulps of the fp64 value."""
    bias_vals = (bias_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    if c_gpu.dtype == torch.float32:
        y_o = oracle.bias_add(oracle.round_to_f32(c_ref), bias_bits).astype(np.float64)
        g = c_gpu.cpu().numpy().astype(np.float64)
        mag = np.maximum(np.abs(g), np.abs(y_o)).astype(np.float32)
        bound = FP32_REL * cabs + np.spacing(mag).astype(np.float64)
        bad = np.abs(g - y_o) > bound
        if bad.any():
            i = tuple(np.argwhere(bad)[0])
            raise AssertionError(f"{what}: {bad.sum()} fp32 outputs out of bound; first {i}: "
                                 f"gpu {g[i]!r} oracle {y_o[i]!r} bound {bound[i]!r}")
        return {"n": int(g.size)}
    gbits = c_gpu.cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    key = bf16_key(oracle.round_to_bf16(c_ref))
    cands = [oracle.bias_add(_bf16_from_key(key + d), bias_bits) for d in (0, -1, 1)]
    exact = gbits == cands[0]
    ok = exact | (gbits == cands[1]) | (gbits == cands[2])
    g = (gbits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    ref = c_ref + bias_vals[None, :]
    near = np.abs(g - ref) <= FP32_REL * cabs + 2 * bf16_ulp(np.maximum(np.abs(c_ref), np.abs(ref)))
    bad = ~ok & ~near
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {bad.sum()} bf16 outputs not admissible; first {i}: gpu {g[i]!r} "
                             f"gemm {c_ref[i]!r} bias {bias_vals[i[1]]!r}")
    return {"exact": int(exact.sum()), "n": int(exact.size)}
