"""Seeded synthetic inputs for the MXFP4 linear path (no quantization arithmetic here).

This module is the one place both the CUDA path's tests/benchmark and the CPU oracle get
their inputs from.  It only draws random numbers and casts them to bf16; it holds none of
the method's arithmetic.

Shapes follow the Flux-12B linears the MXFP4 layers of primus_turbo_mxfp4_local.py are
used for (`MXFP4ColumnParallelLinear` / `MXFP4RowParallelLinear`): 4096 image + 512 text
tokens per micro-batch (4608 rows), hidden size 3072, QKV 3*3072, MLP 4*3072, and the
single-stream block's fused linear1 (3*3072 + 4*3072 = 21504) and linear2 (K = 15360).
No public dataset or checkpoint is involved: every tensor is drawn here from a seed.

Recipe: each tensor is drawn in fp32 on the CPU with torch.Generator(seed) and cast to bf16
with round-to-nearest-even; tensor i of a workload uses seed base_seed + i, in the order
the workload lists them.
"""
from dataclasses import dataclass, field
from typing import Dict, List, Tuple

import numpy as np
import torch


# ---------------------------------------------------------------------------------------
# primitive draws (fp32 on CPU, then one cast to bf16)
# ---------------------------------------------------------------------------------------
def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def normal(shape, std: float, seed: int) -> torch.Tensor:
    """N(0, std^2) in bf16."""
    x = torch.randn(*shape, generator=_gen(seed), dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


def student_t3(shape, scale: float, seed: int) -> torch.Tensor:
    """Student-t with 3 degrees of freedom, z / sqrt(chi2_3 / 3), times `scale`, in bf16."""
    g = _gen(seed)
    z = torch.randn(*shape, generator=g, dtype=torch.float32)
    chi = torch.zeros(*shape, dtype=torch.float32)
    for _ in range(3):
        n = torch.randn(*shape, generator=g, dtype=torch.float32)
        chi.addcmul_(n, n)
    z.div_(torch.sqrt(chi.div_(3.0)))
    if scale != 1.0:
        z.mul_(scale)
    return z.to(torch.bfloat16)


def gelu_like(shape, seed: int) -> torch.Tensor:
    """max(z, 0) + 0.1 * z' with z, z' ~ N(0,1): the skew of a post-GELU activation."""
    g = _gen(seed)
    z = torch.randn(*shape, generator=g, dtype=torch.float32)
    z2 = torch.randn(*shape, generator=g, dtype=torch.float32)
    return (z.clamp_(min=0.0) + 0.1 * z2).to(torch.bfloat16)


def with_outliers_and_zero_blocks(x: torch.Tensor, seed: int, frac: float = 0.01,
                                  factor: float = 50.0, n_row_blocks: int = 2,
                                  n_col_blocks: int = 2) -> torch.Tensor:
    """Multiply `frac` of the entries (chosen by randperm) by `factor`, then zero
    `n_row_blocks` 1x32 blocks along K and `n_col_blocks` 32x1 blocks along M at seeded,
    non-overlapping, 32-aligned positions."""
    g = _gen(seed)
    M, K = x.shape
    y = x.float().reshape(-1)
    n_out = int(round(frac * y.numel()))
    idx = torch.randperm(y.numel(), generator=g)[:n_out]
    y[idx] *= factor
    y = y.reshape(M, K)
    taken = set()
    rows_needed = n_row_blocks + n_col_blocks
    while len(taken) < rows_needed:
        r = int(torch.randint(0, M // 32, (1,), generator=g)) * 32
        c = int(torch.randint(0, K // 32, (1,), generator=g)) * 32
        key = (r // 32, c // 32)
        if key in taken:
            continue
        taken.add(key)
    spots = sorted(taken)
    for i, (rb, cb) in enumerate(spots):
        r, c = rb * 32, cb * 32
        if i < n_row_blocks:
            y[r, c:c + 32] = 0.0          # one rowwise block (row r, 32 columns)
        else:
            y[r:r + 32, c] = 0.0          # one colwise block (32 rows, column c)
    return y.to(torch.bfloat16)


def inject_edge_blocks(x: torch.Tensor, seed: int) -> torch.Tensor:
    """Put MX edge cases at fixed positions of a bf16 tensor, along both packings:
    all-subnormal blocks (bit patterns 0x0001..0x007F, random sign), mixed
    subnormal + normal blocks, near-bf16-max blocks (magnitudes up to 0x7F7F, finite) and
    all-zero blocks.  Each kind is written as a 1x32 row block and as a 32x1 column block.
    """
    g = _gen(seed)
    M, K = x.shape
    bits = x.view(torch.int16).clone()

    def rand_sub(n):
        mag = torch.randint(1, 0x80, (n,), generator=g, dtype=torch.int32)
        sgn = torch.randint(0, 2, (n,), generator=g, dtype=torch.int32) << 15
        return (mag | sgn).to(torch.int32)

    def rand_mixed(n):
        v = rand_sub(n)
        # half of the block: normal values of moderate size (exponent field 100..140)
        ef = torch.randint(100, 141, (n,), generator=g, dtype=torch.int32)
        man = torch.randint(0, 128, (n,), generator=g, dtype=torch.int32)
        sgn = torch.randint(0, 2, (n,), generator=g, dtype=torch.int32) << 15
        normal_bits = sgn | (ef << 7) | man
        pick = torch.arange(n) % 2 == 1
        return torch.where(pick, normal_bits, v)

    def rand_nearmax(n):
        ef = torch.randint(250, 255, (n,), generator=g, dtype=torch.int32)
        man = torch.randint(0, 128, (n,), generator=g, dtype=torch.int32)
        sgn = torch.randint(0, 2, (n,), generator=g, dtype=torch.int32) << 15
        v = sgn | (ef << 7) | man
        v[0] = 0x7F7F  # the largest finite bf16 is always present once
        return v

    def zeros(n):
        return torch.zeros(n, dtype=torch.int32)

    kinds = [rand_sub, rand_mixed, rand_nearmax, zeros]
    nrb, ncb = M // 32, max(K // 32, 1)
    for i, kind in enumerate(kinds):
        # row block: row (7 + 13 i) mod M, columns of block (3 + 5 i) mod (K/32)
        r = (7 + 13 * i) % M
        cb = (3 + 5 * i) % ncb
        c0 = cb * 32
        n = min(32, K - c0)
        bits[r, c0:c0 + n] = _as_i16(kind(32)[:n])
        # column block: rows of block (1 + 3 i) mod (M/32), column (11 + 17 i) mod K
        rb = (1 + 3 * i) % max(nrb, 1)
        c = (11 + 17 * i) % K
        r0 = rb * 32
        n = min(32, M - r0)
        bits[r0:r0 + n, c] = _as_i16(kind(32)[:n])
    return bits.view(torch.bfloat16)


def _as_i16(v32: torch.Tensor) -> torch.Tensor:
    v = v32 & 0xFFFF
    v = torch.where(v >= 0x8000, v - 0x10000, v)
    return v.to(torch.int16)


def bf16_bits(x: torch.Tensor) -> np.ndarray:
    """bf16 tensor (CPU) -> numpy uint16 bit patterns, the oracle's input format."""
    return x.contiguous().view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------------------
@dataclass
class Linear:
    """One MXFP4 linear Y = X . W^T, X[M,K], W[N,K], dY[M,N].  `train` selects the dual
    quantizer and the dgrad/wgrad GEMMs; otherwise the row-only quantizer and the forward
    GEMM alone."""
    name: str
    M: int
    N: int
    K: int
    train: bool
    x_kind: str = "normal"        # "normal" | "gelu_like" | "tiny_outliers"
    w_std: float = 0.02
    dy_std: float = 1e-3

    @property
    def flops_fwd(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def flops_step(self) -> int:
        return self.flops_fwd * (3 if self.train else 1)


@dataclass
class Workload:
    name: str
    description: str
    linears: List[Linear] = field(default_factory=list)
    base_seed: int = 0

    def tensors(self, li: int) -> Dict[str, torch.Tensor]:
        """Draw X, W (and dY when training) of linear li, seeds in that order."""
        lin = self.linears[li]
        s = self.base_seed + 10 * li
        out = {}
        if lin.x_kind == "tiny_outliers":
            out["X"] = with_outliers_and_zero_blocks(normal((lin.M, lin.K), 1.0, s), s + 100)
            out["W"] = with_outliers_and_zero_blocks(normal((lin.N, lin.K), 1.0, s + 1), s + 101)
            if lin.train:
                out["dY"] = normal((lin.M, lin.N), 1.0, s + 2)
            return out
        if lin.x_kind == "gelu_like":
            out["X"] = gelu_like((lin.M, lin.K), s)
        else:
            out["X"] = normal((lin.M, lin.K), 1.0, s)
        out["W"] = normal((lin.N, lin.K), lin.w_std, s + 1)
        if lin.train:
            out["dY"] = normal((lin.M, lin.N), lin.dy_std, s + 2)
        return out


TINY = Workload(
    "tiny_linear_256x256x512",
    "Tiny MXFP4 linear: X[256,512], W[256,512] ~ N(0,1) with 1% x50 outliers and 4 zero "
    "32-blocks each (2 rowwise, 2 colwise); dY[256,256] ~ N(0,1); dual quantize, fwd, "
    "dgrad, wgrad",
    [Linear("tiny", 256, 256, 512, True, "tiny_outliers", 1.0, 1.0)])

FLUX_QKV_FWD = Workload(
    "flux12b_qkv_fwd_4608x9216x3072",
    "Flux-12B joint-block QKV projection, forward only: X[4608,3072] ~ N(0,1), "
    "W[9216,3072] ~ N(0,0.02), row-only quantize, Y[4608,9216] bf16",
    [Linear("qkv", 4608, 9216, 3072, False)])

FLUX_MLP_STEP = Workload(
    "flux12b_mlp_up_train_step_4608x12288x3072",
    "Flux-12B MLP up-projection, full training step: X[4608,3072] ~ N(0,1), "
    "W[12288,3072] ~ N(0,0.02), dY[4608,12288] ~ N(0,1e-3); dual quantize X, W, dY; fwd, "
    "dgrad, wgrad",
    [Linear("mlp_up", 4608, 12288, 3072, True)])

FLUX_SINGLE_BLOCK = Workload(
    "flux12b_single_block_linears_train",
    "Flux-12B single-stream block linear1 X[4608,3072].W1[21504,3072]^T and linear2 "
    "H[4608,15360].W2[3072,15360]^T, fwd+bwd; H GELU-like; weights N(0,0.02); grads "
    "N(0,1e-3)",
    [Linear("linear1", 4608, 21504, 3072, True),
     Linear("linear2", 4608, 3072, 15360, True, "gelu_like")])

SWEEP_M = (4608, 18432, 4600)
SWEEP_K = (3072, 12288, 15360)
SWEEP_SCALE = (1.0, 1e-4, 1e3)


def sweep_tensor(M: int, K: int, scale: float) -> torch.Tensor:
    """One tensor of the quantizer bandwidth/edge sweep: Student-t(3) * scale with the edge
    blocks injected.  Seed derived from the shape and scale index."""
    si = SWEEP_SCALE.index(scale) if scale in SWEEP_SCALE else 9
    seed = 1000 + 100 * si + 10 * (SWEEP_M.index(M) if M in SWEEP_M else 9) + \
        (SWEEP_K.index(K) if K in SWEEP_K else 9)
    x = student_t3((M, K), scale, seed)
    return inject_edge_blocks(x, seed + 50000)


WORKLOADS = {w.name: w for w in (TINY, FLUX_QKV_FWD, FLUX_MLP_STEP, FLUX_SINGLE_BLOCK)}


def quant_sweep_cases() -> List[Tuple[int, int, float]]:
    return [(m, k, s) for m in SWEEP_M for k in SWEEP_K for s in SWEEP_SCALE]
