"""Oracle of the jagged GEMM-Norm backward (fp64, numpy).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``): imported by ``tests/``
and ``bench.py``'s CPU legs, never by the product path.

Source: "Low Precision Flash Attention 4: End-to-End Block-Scaled Attention
for Blackwell", paragraph 4, reports a "jagged GEMM-Norm backward" at 1.76
PFLOP/s, performance-only, and names no operation; paragraph 2 describes the
fused RMSNorm + Quantize and GEMM + Quantize producers with dual scale layouts
and the jagged module (FP8 data unpadded, scales padded to 128-row tiles).

Reading (the plainest operation those words and the rest of the pages fit):
over the T tokens of a jagged batch (sequences concatenated, no padding),
  forward   Y = X W^T               X [T, K], W [N, K]
            r_t = 1 / sqrt(mean_n Y_tn^2 + eps)
            Z_tn = Y_tn r_t gamma_n
  backward  from dZ [T, N]:
            g_tn = gamma_n dZ_tn
            c_t = (1/N) sum_n g_tn Y_tn
            dY_tn = r_t (g_tn - Y_tn r_t^2 c_t)
            dgamma_n = sum_t dZ_tn Y_tn r_t
            dX = dY W,  dW = dY^T X
The MXFP8 path quantizes dY, X and W in 32x32 blocks (transpose-invariant
payloads: one quantization of dY serves both dX, which contracts over N, and
dW, which contracts over T), runs both GEMMs as block-scaled MMAs with fp32
accumulation, and computes dgamma in fp32.  Y arrives as the forward's bf16
output and r as its fp32 rstd; both backward GEMMs take them as given.
"""
from __future__ import annotations

import numpy as np

from . import mx


def forward(x, w, gamma, eps):
    """Exact forward: (Y, r, Z) in fp64."""
    x = np.asarray(x, np.float64); w = np.asarray(w, np.float64)
    y = x @ w.T
    r = 1.0 / np.sqrt((y * y).mean(axis=1) + eps)
    return y, r, y * r[:, None] * np.asarray(gamma, np.float64)[None, :]


def norm_backward(y, r, gamma, dz):
    """dY and dgamma of Z = Y r gamma for given Y, r (fp64)."""
    y = np.asarray(y, np.float64); r = np.asarray(r, np.float64)
    gamma = np.asarray(gamma, np.float64); dz = np.asarray(dz, np.float64)
    g = gamma[None, :] * dz
    c = (g * y).mean(axis=1)
    dy = r[:, None] * (g - y * (r * r * c)[:, None])
    dgamma = (dz * y * r[:, None]).sum(axis=0)
    return dy, dgamma


def backward_exact(x, w, y, r, gamma, dz):
    """Unquantized gradients: (dX, dW, dgamma) in fp64."""
    dy, dgamma = norm_backward(y, r, gamma, dz)
    x = np.asarray(x, np.float64); w = np.asarray(w, np.float64)
    return dy @ w, dy.T @ x, dgamma


def backward_mx(x, w, y, r, gamma, dz):
    """At the method's quantization points: dY, X, W each in 32x32 blocks
    (E4M3 payloads, E8M0 scales; rows past T padded with zeros), then the two
    GEMMs of the dequantized operands (exact in fp64).  Returns
    (dX, dW, dgamma, dY) with dY unquantized."""
    dy, dgamma = norm_backward(y, r, gamma, dz)
    dyq = mx.fake_quant_32x32(dy)
    xq = mx.fake_quant_32x32(np.asarray(x, np.float64))
    wq = mx.fake_quant_32x32(np.asarray(w, np.float64))
    return dyq @ wq, dyq.T @ xq, dgamma, dy


def flops(T, N, K):
    """The two backward GEMMs: 2 * 2 * T * N * K."""
    return 4.0 * T * N * K
