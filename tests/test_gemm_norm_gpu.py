"""Jagged GEMM-Norm backward on the GPU against the oracle.

Three pieces go through the C ABI: the 32x32 quantizer with the payload in
both orientations (lpfa_mx_quantize_t), the RMSNorm backward fused with that
quantization (lpfa_rmsnorm_bwd_mx_quantize, also dgamma), and the two
block-scaled GEMMs dX = dY W, dW = dY^T X (lpfa_mx_gemm, ragged T).

- The plain quantizer is bit-exact against the oracle (payload, its
  transpose, compact scales, both tensor-core scale arrangements).
- dY is computed in fp32 on the GPU and in fp64 by the oracle, so a code may
  differ where the fp32 error can move a value across a rounding midpoint (or
  a block maximum across a power of two).  Each element's error bound eb is
  derived from the fp32 arithmetic; the GPU's code must lie between the
  oracle's codes of dY - eb and dY + eb under the GPU's scale, and its scale
  between the oracle's scales of the block maximum -/+ its bound.
- dX and dW equal the GEMMs of the decoded operands within the fp32
  accumulation bound 1e-5 sum |a||b|, and the oracle's MXFP8 path in relative
  Frobenius norm.
"""
import math

import numpy as np
import pytest
import torch

import workloads
from oracle import gemm_norm as G
from oracle import layouts, mx

pytestmark = pytest.mark.gpu

EPS = 1e-6
U = 2.0 ** -24          # fp32 unit roundoff


@pytest.fixture(scope="module")
def L():
    from mxfp8_block_scaled_quantizer_gb300 import build
    build()
    from mxfp8_block_scaled_quantizer_gb300 import lpfa
    return lpfa


def _np(t):
    return t.cpu().numpy()


def _f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def _padded(x, R):
    Rp = -(-R // 128) * 128
    xp = np.zeros((Rp,) + x.shape[1:])
    xp[:R] = x
    return xp


def _check_layouts(m, R):
    """The transposed payload and both scale arrangements follow from the
    row-major payload and the compact scales."""
    data, sf = _np(m.data), _np(m.sf)
    C = data.shape[1]
    Rp = m.data_t.shape[1]
    dp = np.zeros((Rp, C), np.uint8)
    dp[:R] = data
    assert np.array_equal(_np(m.data_t), dp.T)
    assert np.array_equal(_np(m.sf_mma), layouts.gemm_operand_mma(np.repeat(sf, 32, axis=0)))
    assert np.array_equal(_np(m.sf_mma_t), layouts.gemm_operand_mma(np.repeat(sf.T, 32, axis=0)))


def _check_quant_exact(m, x64, R):
    want = layouts.gemm_quantize(_padded(x64, R), "32x32")
    assert np.array_equal(_np(m.data), want["payload"][:R])
    assert np.array_equal(_np(m.sf), want["sf"])
    assert np.array_equal(_np(m.sf_mma), want["sf_mma"])
    assert np.array_equal(_np(m.sf_mma_t), want["sf_mma_t"])
    _check_layouts(m, R)


@pytest.mark.parametrize("R,C,special", [(300, 384, "inf"), (1, 128, ""), (128, 256, "zero"),
                                         (33, 128, ""), (4097, 512, "")])
def test_quantize_t_bit_exact(L, R, C, special):
    g = torch.Generator().manual_seed(R * 7 + C)
    x = torch.randn(R, C, generator=g) * torch.exp(torch.randn(R, 1, generator=g))
    if special == "inf":
        x[37, 100] = float("inf")
        x[200, 5] = -float("inf")
    if special == "zero":
        x[32:64, 0:32] = 0.0
    x = x.bfloat16()
    m = L.mx_quantize_t(x.cuda())
    torch.cuda.synchronize()
    _check_quant_exact(m, _f64(x), R)


def test_quantize_t_empty_and_bad_arguments(L):
    buf = torch.zeros(256, dtype=torch.uint8, device="cuda")
    p = L._ptr(buf)
    assert L._quant_t(p, 0, 128, p, p, None, None, None, None) == L.LPFA_OK
    assert L._quant_t(p, 1, 96, p, p, None, None, None, None) == L.LPFA_ERR_INVALID_ARG
    assert L._quant_t(None, 1, 128, p, p, None, None, None, None) == L.LPFA_ERR_INVALID_ARG
    assert L._quant_t(buf.data_ptr() + 1, 1, 128, p, p, None, None, None, None) == \
        L.LPFA_ERR_INVALID_ARG


# ------------------------------------------------------------ norm backward
def _dy_bound(y, r, gamma, dz):
    """Per-element bound on |fp32 dY - exact dY| for dY = r (g dZ - Y r^2 c).
    The kernel sums c = mean(g dZ Y) with fused multiply-adds, each lane over
    8 ceil(N/256) terms, then a 5-level butterfly: a chain of at most
    8 ceil(N/256) + 5 roundings, plus the products and the division (the
    bound takes 8 more and a factor 2 of margin)."""
    N = y.shape[1]
    depth = 8 * -(-N // 256) + 13
    gd = np.abs(gamma[None, :] * dz)
    mean_abs = (gd * np.abs(y)).mean(axis=1)
    c = (gamma[None, :] * dz * y).mean(axis=1)
    k2 = np.abs(r * r * c)
    ra = np.abs(r)[:, None]
    eb = ra * (2 * U * gd + 6 * U * np.abs(y) * k2[:, None]
               + np.abs(y) * (r * r)[:, None] * depth * U * mean_abs[:, None])
    dy = ra * np.abs(gamma[None, :] * dz - y * k2[:, None] * np.sign(c)[:, None])
    return 2.0 * (eb + 2 * U * dy)


def _check_open_codes(codes, sf, dy, eb, rows):
    """GPU codes / scales of dY over the given rows (multiple of 32 block
    aligned slice) against the oracle's fp64 dY and bound eb."""
    R, C = dy.shape
    nrb = -(-R // 32)
    dyp = np.zeros((nrb * 32, C)); dyp[:R] = dy
    ebp = np.zeros((nrb * 32, C)); ebp[:R] = eb
    blk = lambda a: a.reshape(nrb, 32, C // 32, 32).transpose(0, 2, 1, 3).reshape(nrb, C // 32, 1024)
    amax = np.abs(blk(dyp)).max(-1)
    ebmax = blk(ebp).max(-1)
    _, lo = mx.scale_exponent(np.maximum(amax - ebmax, 0.0))
    _, hi = mx.scale_exponent(amax + ebmax)
    sf = sf.astype(np.int64)
    assert np.all((lo <= sf) & (sf <= hi))
    open_scales = int(np.sum(lo != hi))
    e = np.repeat(np.repeat(sf - 127, 32, 0), 32, 1)[:R]
    lo_v = mx.e4m3_decode(mx.e4m3_encode(np.ldexp(dy - eb, -e)))
    hi_v = mx.e4m3_decode(mx.e4m3_encode(np.ldexp(dy + eb, -e)))
    got = mx.e4m3_decode(codes)
    assert np.all((lo_v <= got) & (got <= hi_v))
    open_codes = int(np.sum(lo_v != hi_v))
    assert open_codes <= 2e-3 * dy.size + 4
    return open_scales, open_codes


def _norm_inputs(T, N, K, seed):
    inp = workloads.gemm_norm_inputs(T, N, K, seed)
    x64, w64 = _f64(inp["x"]), _f64(inp["w"])
    y, _, _ = G.forward(x64, w64, _f64(inp["gamma"]), EPS)
    y16 = torch.from_numpy(y).to(torch.bfloat16)
    yb = _f64(y16)
    rstd = torch.from_numpy(1.0 / np.sqrt((yb * yb).mean(axis=1) + EPS)).float()
    return inp, y16, rstd


@pytest.mark.parametrize("T,N", [(300, 384), (1, 128), (1000, 256)])
def test_norm_backward_quantize(L, T, N):
    inp, y16, rstd = _norm_inputs(T, N, 256, 11 + T)
    m, dgamma = L.rmsnorm_bwd_mx_quantize(y16.cuda(), inp["dz"].cuda(), inp["gamma"].cuda(),
                                          rstd.cuda())
    torch.cuda.synchronize()
    y, r, gam, dz = _f64(y16), rstd.double().numpy(), _f64(inp["gamma"]), _f64(inp["dz"])
    dy, dg = G.norm_backward(y, r, gam, dz)
    _check_open_codes(_np(m.data), _np(m.sf)[: -(-T // 32)], dy, _dy_bound(y, r, gam, dz), T)
    # padded row blocks are zero blocks
    assert not _np(m.sf)[-(-T // 32):].any()
    _check_layouts(m, T)
    terms = np.abs(dz * y * r[:, None]).sum(axis=0)
    assert np.all(np.abs(_np(dgamma).astype(np.float64) - dg) <= 1e-5 * terms + 1e-30)


# ------------------------------------------------------------ whole backward
def _gemm_bound(a, b):
    return 1e-5 * (np.abs(a) @ np.abs(b)) + 1e-30


def test_backward_ragged(L):
    lengths = workloads.gemm_norm_lengths(6, 1, 400, seed=3)
    T, N, K = int(lengths.sum()), 256, 512
    assert T % 128 != 0
    inp, y16, rstd = _norm_inputs(T, N, K, 21)
    xq = L.mx_quantize_t(inp["x"].cuda())
    wq = L.mx_quantize_t(inp["w"].cuda())
    dx, dw, dgamma = L.gemm_norm_backward(xq, wq, y16.cuda(), rstd.cuda(),
                                          inp["gamma"].cuda(), inp["dz"].cuda())
    dyq, _ = L.rmsnorm_bwd_mx_quantize(y16.cuda(), inp["dz"].cuda(), inp["gamma"].cuda(),
                                       rstd.cuda())
    torch.cuda.synchronize()
    x64, w64 = _f64(inp["x"]), _f64(inp["w"])
    _check_quant_exact(xq, x64, T)
    _check_quant_exact(wq, w64, N)
    dyv = mx.dq_32x32(_np(dyq.data), _np(dyq.sf))
    xv = mx.dq_32x32(_np(xq.data), _np(xq.sf))
    wv = mx.dq_32x32(_np(wq.data), _np(wq.sf))
    gx, gw = _np(dx).astype(np.float64), _np(dw).astype(np.float64)
    assert np.all(np.abs(gx - dyv @ wv) <= _gemm_bound(dyv, wv))
    assert np.all(np.abs(gw - dyv.T @ xv) <= _gemm_bound(dyv.T, xv))
    y, r = _f64(y16), rstd.double().numpy()
    ox, ow, og, _ = G.backward_mx(x64, w64, y, r, _f64(inp["gamma"]), _f64(inp["dz"]))
    rel = lambda a, b: np.linalg.norm(a - b) / np.linalg.norm(b)
    assert rel(gx, ox) < 1e-3 and rel(gw, ow) < 1e-3
    ex = G.backward_exact(x64, w64, y, r, _f64(inp["gamma"]), _f64(inp["dz"]))
    assert 1e-3 < rel(gx, ex[0]) < 0.1 and rel(gw, ex[1]) < 0.1
    terms = np.abs(_f64(inp["dz"]) * y * r[:, None]).sum(axis=0)
    assert np.all(np.abs(_np(dgamma).astype(np.float64) - og) <= 1e-5 * terms + 1e-30)


def test_backward_full_size_sampled(L):
    """The bench's workload (16 jagged sequences, hidden 4096), checked on
    sampled row blocks, rows and entries."""
    cfg = workloads.GEMM_NORM
    lengths = workloads.gemm_norm_lengths(cfg["batch"], cfg["len_min"], cfg["len_max"], cfg["seed"])
    T, N = int(lengths.sum()), cfg["hidden"]
    K = N
    inp = workloads.gemm_norm_inputs(T, N, K, cfg["seed"])
    x, w, gamma, dz = (inp[n].cuda() for n in ("x", "w", "gamma", "dz"))
    y16 = (x @ w.T)                                   # the forward's bf16 Y (input here)
    rstd = torch.rsqrt(y16.float().pow(2).mean(dim=1) + EPS)
    xq = L.mx_quantize_t(x)
    wq = L.mx_quantize_t(w)
    dx, dw, dgamma = L.gemm_norm_backward(xq, wq, y16, rstd, gamma, dz)
    dyq, _ = L.rmsnorm_bwd_mx_quantize(y16, dz, gamma, rstd)
    torch.cuda.synchronize()
    rng = np.random.default_rng(5)
    nrb = -(-T // 32)
    blocks = np.unique(np.concatenate([[0, nrb - 1], rng.integers(0, nrb, 6)]))
    w64, gam = _f64(inp["w"]), _f64(inp["gamma"])
    _check_quant_exact(wq, w64, N)
    wv = mx.dq_32x32(_np(wq.data), _np(wq.sf))
    xsf, dsf = _np(xq.sf), _np(dyq.sf)
    for b in blocks:
        a, e = 32 * b, min(32 * b + 32, T)
        # X: payload rows, their transposed columns and scales
        p, sc = mx.quantize_32x32(_f64(inp["x"][a:e]))
        assert np.array_equal(_np(xq.data[a:e]), p)
        assert np.array_equal(_np(xq.data_t[:, a:e]), p.T)
        assert np.array_equal(xsf[b], sc[0])
        # dY: codes within the fp32 bound
        y, r, dzb = _f64(y16[a:e]), rstd[a:e].double().cpu().numpy(), _f64(inp["dz"][a:e])
        dy, _ = G.norm_backward(y, r, gam, dzb)
        _check_open_codes(_np(dyq.data[a:e]), dsf[b:b + 1], dy, _dy_bound(y, r, gam, dzb), e - a)
        assert np.array_equal(_np(dyq.data_t[:, a:e]), _np(dyq.data[a:e]).T)
    # dX rows: GEMM of the decoded operands
    rows = np.unique(np.concatenate([[0, T - 1], rng.integers(0, T, 14)]))
    for t in rows:
        dyv = mx.e4m3_decode(_np(dyq.data[int(t)])) * mx.e8m0_decode(np.repeat(dsf[t // 32], 32))
        want = dyv @ wv
        got = _np(dx[int(t)]).astype(np.float64)
        assert np.all(np.abs(got - want) <= 1e-5 * (np.abs(dyv) @ np.abs(wv)) + 1e-30)
    # dW entries: contraction over all T tokens
    ns = rng.integers(0, N, 8)
    ks = rng.integers(0, K, 64)
    kt = torch.from_numpy(ks)
    xcols = mx.e4m3_decode(_np(xq.data_t[kt.cuda(), :T])) * \
        mx.e8m0_decode(np.repeat(xsf[:, ks // 32], 32, axis=0)[:T].T)
    for n in ns:
        dcol = mx.e4m3_decode(_np(dyq.data_t[int(n), :T])) * \
            mx.e8m0_decode(np.repeat(dsf[:, n // 32], 32)[:T])
        want = xcols @ dcol
        got = _np(dw[int(n)][kt.cuda()]).astype(np.float64)
        assert np.all(np.abs(got - want) <= 1e-5 * (np.abs(xcols) @ np.abs(dcol)) + 1e-30)
    # dgamma over all tokens, fp64 in row chunks
    dg = np.zeros(N)
    terms = np.zeros(N)
    for a in range(0, T, 8192):
        e = min(a + 8192, T)
        y, r, dzb = _f64(y16[a:e]), rstd[a:e].double().cpu().numpy(), _f64(inp["dz"][a:e])
        pt = dzb * y * r[:, None]
        dg += pt.sum(axis=0)
        terms += np.abs(pt).sum(axis=0)
    assert np.all(np.abs(_np(dgamma).astype(np.float64) - dg) <= 1e-5 * terms + 1e-30)
    assert math.isfinite(float(dx.abs().max())) and math.isfinite(float(dw.abs().max()))
