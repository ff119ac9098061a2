"""Seeded synthetic inputs for the block-scaled quantization workloads.

This module holds no quantization or GEMM arithmetic: it only draws seeded
random bf16 tensors on the CPU with the shapes and value distributions of the
workloads (Gaussian activations with a few large outlier channels, small-std
weights and gradients, sparse 50x outliers for the FP4 case).  Both the CUDA
path and the CPU oracle consume the same tensors.

Seed convention: ``1000 * workload + operand`` with operand A/X = 0, B/W = 1,
G = 2.
"""
from __future__ import annotations

import torch

# Workloads (name -> description); shapes are (rows, cols) of row-major bf16.
WORKLOADS = {
    "mxfp8_gemm_512": "MXFP8 E4M3 GEMM 512x512x512, A N(0,1) with column 7 x 2^12, B N(0,0.02)",
    "mxfp8_quantize_16384x4096": "MXFP8 quantize 16384x4096, N(0,1) + 4 outlier channels 2^10..2^14",
    "mxfp8_linear_8192x4096x14336": "MXFP8 linear layer M=8192 K=4096 N=14336: fprop, dgrad, wgrad",
    "nvfp4_8192": "NVFP4 quantize + GEMM 8192^3, N(0,1) with 0.1% outliers at 50x",
    "deepseek_fp8_4096x7168x2048": "DeepSeek FP8 GEMM M=4096 K=7168 N=2048, 1x128 / 128x128 FP32 scales",
    "mxfp4_8192": "MXFP4 quantize + GEMM 8192^3, N(0,1) with 0.1% outliers at 50x",
}

OUTLIER_COLS_4096 = (5, 1029, 2058, 3087)


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def normal(rows: int, cols: int, std: float, seed: int) -> torch.Tensor:
    """bf16 [rows, cols] drawn from N(0, std^2) in fp32, then rounded to bf16."""
    x = torch.randn(rows, cols, generator=_gen(seed), dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


def with_outlier_channels(rows: int, cols: int, seed: int, channels=None) -> torch.Tensor:
    """N(0,1) activations with 4 outlier channels scaled by 2^(10 + 4j/3), j=0..3
    (2^10 ... 2^14).  Default channel placement spreads them over the hidden
    dimension: columns 5, cols/4+5, cols/2+10, 3cols/4+15 (for cols=4096:
    5, 1029, 2058, 3087)."""
    x = torch.randn(rows, cols, generator=_gen(seed), dtype=torch.float32)
    if channels is None:
        channels = [5, cols // 4 + 5, cols // 2 + 10, 3 * cols // 4 + 15]
        channels = [c % cols for c in channels]
    for j, c in enumerate(channels):
        x[:, c] *= 2.0 ** (10.0 + 4.0 * j / 3.0)
    return x.to(torch.bfloat16)


def with_column_outlier(rows: int, cols: int, seed: int, col: int = 7, factor: float = 2.0 ** 12) -> torch.Tensor:
    """N(0,1) with one outlier channel (column ``col`` scaled by ``factor``)."""
    x = torch.randn(rows, cols, generator=_gen(seed), dtype=torch.float32)
    if cols > col:
        x[:, col] *= factor
    return x.to(torch.bfloat16)


def with_sparse_outliers(rows: int, cols: int, seed: int, p: float = 0.001, factor: float = 50.0) -> torch.Tensor:
    """N(0,1) where a Bernoulli(p) mask of elements is multiplied by ``factor``."""
    g = _gen(seed)
    x = torch.randn(rows, cols, generator=g, dtype=torch.float32)
    mask = torch.rand(rows, cols, generator=g) < p
    x[mask] *= factor
    return x.to(torch.bfloat16)


# ------------------------------------------------------------ workloads
def mxfp8_gemm_512(M=512, N=512, K=512):
    a = with_column_outlier(M, K, 1000)
    b = normal(N, K, 0.02, 1001)
    return a, b


def mxfp8_quantize(rows=16384, cols=4096):
    return with_outlier_channels(rows, cols, 2000)


def mxfp8_linear(M=8192, K=4096, N=14336):
    x = normal(M, K, 1.0, 3000)
    w = normal(N, K, 0.02, 3001)
    g = normal(M, N, 1e-3, 3002)
    return x, w, g


def nvfp4_pair(M=8192, N=8192, K=8192):
    a = with_sparse_outliers(M, K, 4000)
    b = with_sparse_outliers(N, K, 4001)
    return a, b


def mxfp4_pair(M=8192, N=8192, K=8192):
    """MXFP4 product operands: the NVFP4 recipe (N(0,1) with 0.1% of elements x50), own seeds."""
    return with_sparse_outliers(M, K, 6000), with_sparse_outliers(N, K, 6001)


def deepseek_pair(M=4096, N=2048, K=7168):
    a = normal(M, K, 1.0, 5000)
    b = normal(N, K, 0.02, 5001)
    return a, b


def bf16_bits(x: torch.Tensor):
    """bf16 tensor -> numpy uint16 view of its bit patterns (CPU)."""
    import numpy as np
    return x.contiguous().view(torch.int16).numpy().view(np.uint16)
