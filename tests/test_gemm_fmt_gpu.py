"""Block-scaled GEMM on MXFP6 / MXFP4 / E5M2 operands (kind::mxf8f6f4).

Each operand goes through the product path: lpfa_mx_quantize_fmt (1x32
blocks along K), lpfa_mx_pack_operand (the tensor core's byte layout), then
lpfa_mx_gemm_fmt.  Checked against the oracle: the packed bytes equal the
oracle's layout of the oracle's codes bit for bit, and D equals the oracle's
GEMM of the decoded operands (every product exact in fp64) within the fp32
accumulation bound 1e-5 of sum |a||b|."""
import numpy as np
import pytest
import torch

from oracle import layouts, mx

pytestmark = pytest.mark.gpu

FMT = {"e4m3": 0, "e5m2": 1, "e3m2": 2, "e2m3": 3, "e2m1": 4}


@pytest.fixture(scope="module")
def L():
    from mxfp8_block_scaled_quantizer_gb300 import build
    build()
    from mxfp8_block_scaled_quantizer_gb300 import lpfa
    return lpfa


def _operand(L, x, fmt):
    """bf16 [R, K] -> (packed operand bytes, tensor-core scales, oracle codes,
    oracle scale codes)."""
    R, K = x.shape
    m = L.mx_quantize(x.view(R, K // 128, 128).cuda(), L.LPFA_BLK_1X32,
                      L.dense_seqs(1, R), compact=True, fmt=FMT[fmt])
    packed = L.mx_pack_operand(m.data.view(R, K), FMT[fmt])
    codes, sc = mx.quantize_1x32(x.float().numpy().astype(np.float64), fmt)
    torch.cuda.synchronize()
    assert np.array_equal(m.data.view(R, K).cpu().numpy(), codes)
    assert np.array_equal(packed.cpu().numpy(), layouts.mma_operand_bytes(codes, fmt))
    return packed, m.sf_mma, codes, sc


@pytest.mark.parametrize("fa,fb", [("e5m2", "e4m3"), ("e3m2", "e2m3"), ("e2m3", "e4m3"),
                                   ("e2m1", "e2m1"), ("e2m1", "e5m2"), ("e3m2", "e3m2"),
                                   ("e4m3", "e2m1")])
def test_gemm_element_formats(L, fa, fb):
    M, N, K = 256, 512, 512
    g = torch.Generator().manual_seed(len(fa + fb) * 7 + FMT[fa] * 5 + FMT[fb])
    xa = (torch.randn(M, K, generator=g) * torch.exp(torch.randn(M, 1, generator=g))).bfloat16()
    xb = (torch.randn(N, K, generator=g) * torch.exp(torch.randn(1, K, generator=g))).bfloat16()
    pa, sfa, ca, sa = _operand(L, xa, fa)
    pb, sfb, cb, sb = _operand(L, xb, fb)
    d = torch.empty((M, N), dtype=torch.float32, device="cuda")
    L.lpfa_mx_gemm_fmt(pa, sfa, pb, sfb, d, FMT[fa], FMT[fb])
    torch.cuda.synchronize()
    want = mx.mx_gemm(ca, sa, cb, sb, fa, fb)
    bound = 1e-5 * (np.abs(mx.dq_1x32(ca, sa, fa)) @ np.abs(mx.dq_1x32(cb, sb, fb)).T)
    got = d.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - want) <= bound + 1e-30)
    assert np.abs(want).max() > 0


def test_pack_rejects_bad_arguments(L):
    import ctypes
    buf = torch.zeros((2, 32), dtype=torch.uint8, device="cuda")
    assert L._pack_operand(L._ptr(buf), 2, 24, 4, L._ptr(buf), None) == L.LPFA_ERR_INVALID_ARG
    assert L._pack_operand(L._ptr(buf), 2, 32, 9, L._ptr(buf), None) == L.LPFA_ERR_INVALID_ARG
    assert L._pack_operand(None, 2, 32, 4, L._ptr(buf), None) == L.LPFA_ERR_INVALID_ARG
