"""RMSNorm followed by MX quantization: the fused producer named in "Low
Precision Flash Attention 4: End-to-End Block-Scaled Attention for Blackwell",
paragraph 2 (fused RMSNorm+Quantize kernels that emit FP8 output with dual
scale factor layouts in one pass).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Definition (the pages name the operation and give no formula): for each token
row x of N = H * D values and a weight vector w of N values,

    y = x / sqrt(mean(x^2) + eps) * w,

then y [T, H, D] is quantized exactly as the quantizer quantizes its bf16
input (``layouts.oracle_quantize``: 1x32, 32 along tokens or 32x32 blocks,
compact and tensor-core scale layouts).  ``rmsnorm_fp64`` is that definition
in fp64.

Reading (where the pages are silent, listed in the design notes): the E4M3
codes and E8M0 scales are integers decided from y, so both sides decide them
on the same fp32 values, formed as

    ss    = sum of the squares x_i^2 in fp32 (each square is exact: x is
            bf16), accumulated in a fixed order: partial sum l (l = 0..31)
            runs over the 8-element chunks l, l + 32, l + 64, ... of the row,
            element by element; the 32 partial sums are combined pairwise at
            index distance 16, 8, 4, 2, 1 (every fp32 addition rounds to
            nearest even);
    rstd  = 1 / sqrt(ss / N + eps), each operation correctly rounded in fp32;
    y     = (x * rstd) * w, each product rounded to fp32.

``rmsnorm_fp32`` computes that sequence with numpy float32 scalars and arrays
(IEEE operations, no fused multiply-add); the pins in
``tests/test_oracle_norm.py`` tie it to ``rmsnorm_fp64`` within fp32 rounding
and to closed forms.
"""
from __future__ import annotations

import numpy as np

from . import layouts


def rmsnorm_fp64(x, w, eps) -> np.ndarray:
    """The plain definition in fp64: x [T, N], w [N] -> y [T, N]."""
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + float(eps)) * w


def _sum_squares_fp32(row: np.ndarray) -> np.float32:
    """Sum of squares of one fp32 row in the fixed order of the reading."""
    n = row.shape[0]
    chunks = row.reshape(n // 8, 8)
    part = np.zeros(32, dtype=np.float32)
    for c in range(n // 8):
        l = c % 32
        for k in range(8):
            v = chunks[c, k]
            part[l] = np.float32(part[l] + np.float32(v * v))
    for dist in (16, 8, 4, 2, 1):
        part = (part + part[np.arange(32) ^ dist]).astype(np.float32)
    return part[0]


def rmsnorm_fp32(x, w, eps) -> tuple:
    """The fp32 sequence of the reading: x [T, N] (bf16 values), w [N] (bf16
    values), eps > 0.  Returns (y float32 [T, N], rstd float32 [T])."""
    x = np.asarray(x, dtype=np.float32)
    w = np.asarray(w, dtype=np.float32)
    T, n = x.shape
    assert n % 8 == 0
    eps32 = np.float32(eps)
    nf = np.float32(n)
    rstd = np.zeros(T, dtype=np.float32)
    with np.errstate(over="ignore", invalid="ignore", divide="ignore"):
        for t in range(T):
            ss = _sum_squares_fp32(x[t])
            r = np.float32(np.float32(1.0) / np.sqrt(np.float32(np.float32(ss / nf) + eps32)))
            rstd[t] = r
        y = ((x * rstd[:, None]).astype(np.float32) * w[None, :]).astype(np.float32)
    return y, rstd


def rms_quantize(x, w, eps, heads, cu_seqlens, block) -> dict:
    """Oracle of the fused producer: x [T, heads * D] bf16 values, w [heads *
    D].  Returns the quantizer's outputs for y (payload, sf, sf_mma,
    sf_mma_t) plus rstd [T]."""
    x = np.asarray(x, dtype=np.float32)
    T, n = x.shape
    y, rstd = rmsnorm_fp32(x, w, eps)
    out = layouts.oracle_quantize(y.astype(np.float64).reshape(T, heads, n // heads),
                                  cu_seqlens, block)
    out["rstd"] = rstd
    return out
