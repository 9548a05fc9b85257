"""Pins for the GEMM-Norm backward oracle (CPU only).

The exact backward is checked against torch autograd in fp64 (a library
routine, independent of the oracle's hand-derived formula): the norm's
gradient w.r.t. Y and gamma, and the whole chain X, W -> Y -> Z.  The MXFP8
path is restated here with a brute-force 32x32 block rounding (torch's E4M3
decoder, exhaustive nearest search), not the oracle's codec.
"""
import math

import numpy as np
import torch

from oracle import gemm_norm as G

_GRID = torch.arange(0, 127, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
_EVEN = (np.arange(127) % 2) == 0


def _round_block(blk):
    amax = float(np.abs(blk).max())
    if amax == 0.0:
        return np.zeros_like(blk)
    e = math.frexp(amax)[1] - 1 - 8
    a = blk * 2.0 ** -e
    mag = np.minimum(np.abs(a), 448.0)
    d = np.abs(mag[..., None] - _GRID)
    cand = d == d.min(axis=-1, keepdims=True)
    even = cand & _EVEN
    pick = np.where(even.any(-1), even.argmax(-1), cand.argmax(-1))
    return np.sign(a) * _GRID[pick] * 2.0 ** e


def _blocks_32x32(x):
    R, C = x.shape
    Rp = -(-R // 32) * 32
    xp = np.zeros((Rp, C)); xp[:R] = x
    out = np.empty_like(xp)
    for r in range(0, Rp, 32):
        for c in range(0, C, 32):
            out[r:r + 32, c:c + 32] = _round_block(xp[r:r + 32, c:c + 32])
    return out[:R]


def _inputs(rng, T=70, N=64, K=96):
    x = rng.standard_normal((T, K))
    w = rng.standard_normal((N, K)) / math.sqrt(K)
    gamma = 1.0 + 0.1 * rng.standard_normal(N)
    dz = rng.standard_normal((T, N))
    return x, w, gamma, dz


def test_norm_backward_matches_autograd(rng):
    x, w, gamma, dz = _inputs(rng)
    y = x @ w.T
    yt = torch.from_numpy(y).requires_grad_(True)
    gt = torch.from_numpy(gamma).requires_grad_(True)
    eps = 1e-5
    z = yt * torch.rsqrt((yt * yt).mean(dim=1, keepdim=True) + eps) * gt
    z.backward(torch.from_numpy(dz))
    r = 1.0 / np.sqrt((y * y).mean(axis=1) + eps)
    dy, dgamma = G.norm_backward(y, r, gamma, dz)
    assert np.allclose(dy, yt.grad.numpy(), rtol=1e-10, atol=1e-12)
    assert np.allclose(dgamma, gt.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_full_backward_matches_autograd(rng):
    x, w, gamma, dz = _inputs(rng)
    eps = 1e-6
    xt = torch.from_numpy(x).requires_grad_(True)
    wt = torch.from_numpy(w).requires_grad_(True)
    gt = torch.from_numpy(gamma).requires_grad_(True)
    yt = xt @ wt.T
    zt = yt * torch.rsqrt((yt * yt).mean(dim=1, keepdim=True) + eps) * gt
    zt.backward(torch.from_numpy(dz))
    y, r, z = G.forward(x, w, gamma, eps)
    assert np.allclose(z, zt.detach().numpy(), rtol=1e-12, atol=1e-12)
    dx, dw, dgamma = G.backward_exact(x, w, y, r, gamma, dz)
    assert np.allclose(dx, xt.grad.numpy(), rtol=1e-9, atol=1e-12)
    assert np.allclose(dw, wt.grad.numpy(), rtol=1e-9, atol=1e-12)
    assert np.allclose(dgamma, gt.grad.numpy(), rtol=1e-9, atol=1e-12)


def test_mx_path_restated(rng):
    """dX = Q(dY) Q(W), dW = Q(dY)^T Q(X) with Q the 32x32 block rounding;
    the quantization really changes the result."""
    x, w, gamma, dz = _inputs(rng, T=70, N=64, K=96)
    y, r, _ = G.forward(x, w, gamma, 1e-6)
    dx, dw, dgamma, dy = G.backward_mx(x, w, y, r, gamma, dz)
    dyq, xq, wq = _blocks_32x32(dy), _blocks_32x32(x), _blocks_32x32(w)
    assert np.allclose(dx, dyq @ wq, rtol=1e-12, atol=1e-14)
    assert np.allclose(dw, dyq.T @ xq, rtol=1e-12, atol=1e-14)
    ex = G.backward_exact(x, w, y, r, gamma, dz)
    rel = np.linalg.norm(dx - ex[0]) / np.linalg.norm(ex[0])
    assert 1e-3 < rel < 0.1
    assert np.array_equal(dgamma, ex[2])
