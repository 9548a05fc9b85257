"""Fused RMSNorm + MX quantization on the GPU: E4M3 payloads, E8M0 scales
(compact and both tensor-core arrangements) and rstd bit-exact against the
oracle (``oracle/norm.py``) on ragged, jagged and full-size inputs and on edge
rows.  The operation is the fused producer of "Low Precision Flash Attention
4: End-to-End Block-Scaled Attention for Blackwell", paragraph 2."""
import numpy as np
import pytest
import torch

from oracle import norm

pytestmark = pytest.mark.gpu

BLOCKS = {"1x32": 0, "32x32": 2}
EPS = 1e-6


@pytest.fixture(scope="module")
def L():
    from mxfp8_block_scaled_quantizer_gb300 import build
    build()
    from mxfp8_block_scaled_quantizer_gb300 import lpfa
    assert lpfa.lpfa_device_supported()
    return lpfa


def _inputs(T, H, D, seed):
    g = torch.Generator().manual_seed(seed)
    x = (torch.randn(T, H, D, generator=g) * torch.exp(0.5 * torch.randn(T, 1, 1, generator=g)))
    w = 1.0 + 0.1 * torch.randn(H * D, generator=g)
    return x.bfloat16(), w.bfloat16()


def _run(L, x, w, cu, block):
    seqs = L.varlen_seqs(torch.as_tensor(cu, dtype=torch.int32).cuda())
    m, rstd = L.rmsnorm_mx_quantize(x.cuda(), w.cuda(), EPS, BLOCKS[block], seqs)
    torch.cuda.synchronize()
    got = {k: (None if getattr(m, k) is None else getattr(m, k).cpu().numpy())
           for k in ("data", "sf", "sf_mma", "sf_mma_t")}
    got["rstd"] = rstd.cpu().numpy()
    return got


def _check(got, x, w, cu, block, tag):
    T, H, D = x.shape
    want = norm.rms_quantize(x.float().numpy().reshape(T, H * D), w.float().numpy(), EPS, H,
                             np.asarray(cu), block)
    g, r = got["rstd"], want["rstd"]
    assert np.array_equal(np.isnan(g), np.isnan(r)), f"{tag}: rstd NaN rows"
    ok = ~np.isnan(r)
    assert np.array_equal(g[ok].view(np.uint32), r[ok].view(np.uint32)), f"{tag}: rstd"
    assert np.array_equal(got["data"], want["payload"]), f"{tag}: payload"
    assert np.array_equal(got["sf"], want["sf"]), f"{tag}: compact scales"
    assert np.array_equal(got["sf_mma"], want["sf_mma"]), f"{tag}: mma scales"
    if want["sf_mma_t"] is not None:
        assert np.array_equal(got["sf_mma_t"], want["sf_mma_t"]), f"{tag}: mma_t"


@pytest.mark.parametrize("block", list(BLOCKS))
@pytest.mark.parametrize("H,D", [(4, 128), (6, 64), (3, 128)])
def test_ragged_dense(L, block, H, D):
    """One sequence of 300 tokens: several 32-row blocks and a ragged tail."""
    x, w = _inputs(300, H, D, seed=H * D)
    cu = [0, 300]
    _check(_run(L, x, w, cu, block), x, w, cu, block, f"T300 H{H} D{D}")


@pytest.mark.parametrize("block", list(BLOCKS))
def test_jagged(L, block):
    """Packed sequences of uneven lengths (scale rows padded per sequence)."""
    lens = [1, 130, 31, 257, 64]
    cu = np.concatenate([[0], np.cumsum(lens)])
    x, w = _inputs(int(cu[-1]), 8, 128, seed=11)
    _check(_run(L, x, w, cu, block), x, w, cu, block, "jagged")


@pytest.mark.parametrize("block", list(BLOCKS))
def test_edge_rows(L, block):
    """Zero rows (rstd = 1/sqrt(eps)), a NaN (its blocks get code 0xFF and
    payload 0x7F), a value whose square overflows fp32 (rstd = 0: y = 0),
    subnormal-range inputs and a saturating outlier."""
    x, w = _inputs(96, 4, 128, seed=5)
    x[0] = 0.0
    x[33, 1, 7] = float("nan")
    x[40, 2, 0] = 2.0 ** 70
    x[64] = x[64] * 2.0 ** -120
    x[70, 0, 3] = 3.0e4
    cu = [0, 96]
    _check(_run(L, x, w, cu, block), x, w, cu, block, "edges")


@pytest.mark.parametrize("block", list(BLOCKS))
def test_full_size_sampled(L, block):
    """The bench's launch: x [65536, 32, 128] (8 sequences of 8192 tokens,
    hidden 4096); three 128-token slices (every scale tile they own)
    against the oracle run on the slice alone."""
    T, H, D = 8 * 8192, 32, 128
    x, w = _inputs(T, H, D, seed=2)
    seqs = L.dense_seqs(8, 8192)
    m, rstd = L.rmsnorm_mx_quantize(x.cuda(), w.cuda(), EPS, BLOCKS[block], seqs)
    torch.cuda.synchronize()
    for a in (0, 8192 * 3 + 4096, T - 128):
        xs = x[a:a + 128]
        got = {"data": m.data[a:a + 128].cpu().numpy(), "rstd": rstd[a:a + 128].cpu().numpy(),
               "sf_mma": m.sf_mma[a // 128:a // 128 + 1].cpu().numpy(),
               "sf_mma_t": None if m.sf_mma_t is None else m.sf_mma_t[a // 128:a // 128 + 1].cpu().numpy()}
        if block == "1x32":
            got["sf"] = m.sf[a:a + 128].cpu().numpy()
        else:
            got["sf"] = m.sf[a // 32:a // 32 + 4].cpu().numpy()
        _check(got, xs, w, [0, 128], block, f"slice {a}")


def test_rejects_bad_arguments(L):
    x, w = _inputs(64, 2, 128, seed=1)
    seqs = L.dense_seqs(1, 64)
    xc, wc = x.cuda(), w.cuda()
    out = torch.empty((64, 2, 128), dtype=torch.uint8, device="cuda")
    with pytest.raises(L.LpfaError):
        L.lpfa_rmsnorm_mx_quantize(seqs, xc, wc, 0.0, 0, out)
    with pytest.raises(L.LpfaError):
        L.lpfa_rmsnorm_mx_quantize(seqs, xc, wc, 1e-6, 1, out)   # 32x1: unsupported
