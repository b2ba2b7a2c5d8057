"""GB300-native MXFP4 linear hot path: the dual / row-only block-scaled quantizer and the
tcgen05 block-scaled MXF4 GEMM, behind a small C ABI (include/mxfp4.h).

Importing the package loads nothing; `mxfp4_block_scaled_quantize_gb300.abi` loads the
CUDA library and raises if it has not been built.
"""
__all__ = ["abi", "workloads"]
