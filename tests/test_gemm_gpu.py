"""Block-scaled MXFP8 GEMM (tcgen05) against the oracle's MX GEMM: every
product of decoded operands is exact, so the only difference is fp32
accumulation order."""
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


def _gemm_sf_layout(sc):
    """[R, K/32] compact scales -> [R/128][K/128][512] tensor-core tiles."""
    R, nk = sc.shape
    out = np.zeros((R // 128, nk // 4, 512), dtype=np.uint8)
    r, kb = np.meshgrid(np.arange(R), np.arange(nk), indexing="ij")
    out[r // 128, kb // 4, layouts.atom_offset(r % 128, kb % 4)] = sc[r, kb]
    return out


@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (256, 512, 512),
                                   (384, 768, 1024)])
def test_mx_gemm_matches_oracle(L, M, N, K):
    rng = np.random.default_rng(M + N + K)
    a = rng.standard_normal((M, K)) * np.exp(rng.uniform(-4, 4, (M, 1)))
    b = rng.standard_normal((N, K)) * np.exp(rng.uniform(-4, 4, (1, K)))
    pa, sa = mx.quantize_1x32(a)
    pb, sb = mx.quantize_1x32(b)
    want = mx.mx_gemm(pa, sa, pb, sb)
    dev = lambda z: torch.from_numpy(np.ascontiguousarray(z)).cuda()
    d = torch.empty((M, N), dtype=torch.float32, device="cuda")
    L.lpfa_mx_gemm(dev(pa), dev(_gemm_sf_layout(sa)), dev(pb),
                   dev(_gemm_sf_layout(sb)), d)
    torch.cuda.synchronize()
    got = d.cpu().numpy().astype(np.float64)
    scale = np.abs(mx.dq_1x32(pa, sa)) @ np.abs(mx.dq_1x32(pb, sb)).T
    assert np.all(np.abs(got - want) <= 1e-5 * scale + 1e-30)
