"""Dense FP4 GEMM (kind::mxf4nvf4) with MXFP4 and NVFP4 scales, and the
NVFP4 quantizer, against the oracle.

The NVFP4 quantizer must reproduce the oracle's codes and scales bit for bit
(its divisions are single fp32 divisions on both sides); the dense packing and
the tensor-core scale tiles equal the oracle's layouts; D equals the oracle's
GEMM of the decoded operands (every product exact in fp64) within the fp32
accumulation bound 1e-5 of sum |a||b|."""
import numpy as np
import pytest
import torch

from oracle import layouts, mx

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    from mxfp8_block_scaled_quantizer_gb300 import build
    build()
    from mxfp8_block_scaled_quantizer_gb300 import lpfa
    return lpfa


def _inputs(M, N, K, seed):
    g = torch.Generator().manual_seed(seed)
    xa = (torch.randn(M, K, generator=g) * torch.exp(torch.randn(M, 1, generator=g))).bfloat16()
    xb = (torch.randn(N, K, generator=g) * torch.exp(torch.randn(1, K, generator=g))).bfloat16()
    return xa, xb


def _check(d, want, absprod):
    got = d.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - want) <= 1e-5 * absprod + 1e-30)
    assert np.abs(want).max() > 0


def test_nvfp4_quantizer_bit_exact(L):
    x = _inputs(256, 128, 320, seed=3)[0]
    x[5, :16] = 0.0                                   # an all-zero block
    x[9, 32:48] *= 1e-4                               # tiny scales
    out, sf, mma = L.nvfp4_quantize(x.cuda())
    torch.cuda.synchronize()
    codes, sc = mx.quantize_nvfp4(x.float().numpy())
    assert np.array_equal(sf.cpu().numpy(), sc)
    assert np.array_equal(out.cpu().numpy(), layouts.fp4_dense_bytes(codes))
    assert np.array_equal(mma.cpu().numpy(), layouts.gemm_operand_mma(sc))


@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (256, 512, 1024)])
def test_mxfp4_gemm(L, M, N, K):
    xa, xb = _inputs(M, N, K, seed=M + K)

    def operand(x):
        R = x.shape[0]
        m = L.mx_quantize(x.view(R, K // 128, 128).cuda(), L.LPFA_BLK_1X32,
                          L.dense_seqs(1, R), compact=True, fmt=L.LPFA_ELEM_E2M1)
        dense = L.fp4_pack_dense(m.data.view(R, K))
        codes, sc = mx.quantize_1x32(x.float().numpy().astype(np.float64), "e2m1")
        return dense, m.sf_mma, codes, sc

    pa, sfa, ca, sa = operand(xa)
    pb, sfb, cb, sb = operand(xb)
    d = torch.empty((M, N), dtype=torch.float32, device="cuda")
    L.lpfa_mx_gemm_fp4(pa, sfa, pb, sfb, d, nvfp4=False)
    torch.cuda.synchronize()
    assert np.array_equal(pa.cpu().numpy(), layouts.fp4_dense_bytes(ca))
    want = mx.fp4_gemm(ca, sa, cb, sb, "mx")
    absprod = np.abs(mx.dq_1x32(ca, sa, "e2m1")) @ np.abs(mx.dq_1x32(cb, sb, "e2m1")).T
    _check(d, want, absprod)


@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (256, 512, 1024)])
def test_nvfp4_gemm(L, M, N, K):
    xa, xb = _inputs(M, N, K, seed=M + K + 1)
    pa, _, sfa = L.nvfp4_quantize(xa.cuda())
    pb, _, sfb = L.nvfp4_quantize(xb.cuda())
    d = torch.empty((M, N), dtype=torch.float32, device="cuda")
    L.lpfa_mx_gemm_fp4(pa, sfa, pb, sfb, d, nvfp4=True)
    torch.cuda.synchronize()
    ca, sa = mx.quantize_nvfp4(xa.float().numpy())
    cb, sb = mx.quantize_nvfp4(xb.float().numpy())
    want = mx.fp4_gemm(ca, sa, cb, sb, "nv")
    absprod = np.abs(mx.dq_nvfp4(ca, sa)) @ np.abs(mx.dq_nvfp4(cb, sb)).T
    _check(d, want, absprod)
