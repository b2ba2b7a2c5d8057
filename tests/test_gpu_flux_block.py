"""GPU parity of the Flux-12B single-stream block's linears, the largest Flux config:
linear1 X[4608,3072] . W1[21504,3072]^T and linear2 H[4608,15360] . W2[3072,15360]^T with
H GELU-like (max(z,0) + 0.1 z'), weights N(0,0.02), grads N(0,1e-3), each run forward and
backward (fwd, dgrad dX = dY . W, wgrad dW = dY^T . X) in the launch configuration of the
benchmark's step (MXFP4Block: forwards in order, backwards in reverse order).

Every blob the step quantizes is compared byte for byte with the oracle on sampled rows and
whole sampled columns; every GEMM output on sampled rows against the fp64 oracle, once with
bf16 and once with fp32 outputs, so the strict fp32 bound 1e-5 * sum|ab| covers each
full-size backward shape.
"""
import functools

import numpy as np
import pytest
import torch

import oracle
from mxfp4_block_scaled_quantize_gb300 import abi, workloads
from mxfp4_block_scaled_quantize_gb300.linear import MXFP4Block
from parity import check_gemm, check_quantized_sampled

pytestmark = pytest.mark.gpu

WL = workloads.FLUX_SINGLE_BLOCK


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield
    block_outputs.cache_clear()
    assert abi.mxfp4_last_device_error() == abi.MXFP4_OK


@functools.lru_cache(maxsize=None)
def host_tensors(li):
    return WL.tensors(li)


@functools.lru_cache(maxsize=None)
def bits(li, name):
    return workloads.bf16_bits(host_tensors(li)[name])


@functools.lru_cache(maxsize=None)
def block_outputs(out_dtype):
    """Runs one step of the block; returns per linear (Y, dX, dW) and the layers (for their
    blobs), all on the GPU."""
    inputs = [{k: v.cuda() for k, v in host_tensors(i).items()} for i in range(len(WL.linears))]
    blk = MXFP4Block([(l.name, l.M, l.N, l.K) for l in WL.linears], train=True, out_dtype=out_dtype)
    outs = blk.step(inputs)
    torch.cuda.synchronize()
    assert abi.mxfp4_last_device_error() == abi.MXFP4_OK
    return outs, blk.layers


def sample(n, count, seed):
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([rng.choice(n, count, replace=False), [0, 127, 128, n - 1]]))


@functools.lru_cache(maxsize=None)
def oracle_rows(li, which):
    """(sampled output rows, C[rows], sum|ab|[rows]) of GEMM `which` of linear li."""
    lin = WL.linears[li]
    x, w, dy = bits(li, "X"), bits(li, "W"), bits(li, "dY")
    if which == "fwd":          # Y rows: X rows against the row blob of W
        rows = sample(lin.M, 8, 10 + li)
        aq, a_s = oracle.quantize_row(np.ascontiguousarray(x[rows]))
        bq, b_s = oracle.quantize_row(w)
    elif which == "dgrad":      # dX rows: dY rows against the col blob of W
        rows = sample(lin.M, 8, 20 + li)
        aq, a_s = oracle.quantize_row(np.ascontiguousarray(dy[rows]))
        bq, b_s = oracle.quantize_col(w)
    else:                       # dW row n: column n of dY against the col blob of X
        rows = sample(lin.N, 8, 30 + li)
        aq, a_s = oracle.quantize_col(np.ascontiguousarray(dy[:, rows]))
        bq, b_s = oracle.quantize_col(x)
    c, cabs = oracle.gemm(aq, a_s, bq, b_s)
    return rows, c, cabs


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("which", ["fwd", "dgrad", "wgrad"])
@pytest.mark.parametrize("li", [0, 1], ids=["linear1", "linear2"])
def test_block_gemm_sampled(li, which, out_dtype):
    outs, _ = block_outputs(out_dtype)
    got = outs[li][("fwd", "dgrad", "wgrad").index(which)]
    rows, c, cabs = oracle_rows(li, which)
    lin = WL.linears[li]
    check_gemm(got[torch.as_tensor(rows, device="cuda")], c, cabs,
               f"flux single block {lin.name} {which} {str(out_dtype)[6:]}")


@pytest.mark.parametrize("li", [0, 1], ids=["linear1", "linear2"])
def test_block_blobs_sampled(li):
    # The dual blobs of X (H for linear2, the GELU-skewed activation), W and dY that the
    # step's GEMMs consumed, byte for byte against the oracle.
    _, layers = block_outputs(torch.bfloat16)
    L = layers[li]
    t = host_tensors(li)
    name = "H" if li == 1 else "X"
    check_quantized_sampled(t["X"], L.x_row + L.x_col, True, f"{WL.linears[li].name} {name}", seed=li)
    check_quantized_sampled(t["W"], L.w_row + L.w_col, True, f"{WL.linears[li].name} W", n_rows=24,
                            n_cols=24, seed=li + 2)
    check_quantized_sampled(t["dY"], L.dy_row + L.dy_col, True, f"{WL.linears[li].name} dY", n_rows=24,
                            n_cols=24, seed=li + 4)
