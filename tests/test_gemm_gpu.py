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
    out = np.zeros((-(-R // 128), nk // 4, 512), dtype=np.uint8)
    r, kb = np.meshgrid(np.arange(R), np.arange(nk), indexing="ij")
    out[r // 128, kb // 4, layouts.atom_offset(r % 128, kb % 4)] = sc[r, kb]
    return out


@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (256, 512, 512),
                                   (384, 768, 1024), (1000, 512, 256), (2560, 2048, 512)])
def test_mx_gemm_matches_oracle(L, M, N, K):
    """CTA-pair tiles of 256 rows: a half-empty pair (M = 128, 384), a ragged
    M and more tiles than resident pairs."""
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


# ------------------------------------------------------ quantizing epilogue
def _operands(M, N, K, seed):
    rng = np.random.default_rng(seed)
    a = rng.standard_normal((M, K)) * np.exp(rng.uniform(-3, 3, (M, 1)))
    b = rng.standard_normal((N, K)) * np.exp(rng.uniform(-3, 3, (1, K)))
    pa, sa = mx.quantize_1x32(a)
    pb, sb = mx.quantize_1x32(b)
    return pa, sa, pb, sb


def _dev(z):
    return torch.from_numpy(np.ascontiguousarray(z)).cuda()


@pytest.mark.parametrize("block", ["1x32", "32x32"])
@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (384, 768, 512), (512, 1024, 256)])
def test_mx_gemm_quantize_matches_oracle(L, block, M, N, K):
    """The fused output equals the oracle's quantization of the kernel's own
    fp32 result bit for bit (the codes are decided on those values), and the
    fp32 result is the GEMM within fp32 accumulation error."""
    pa, sa, pb, sb = _operands(M, N, K, seed=M + N + K)
    blk = {"1x32": L.LPFA_BLK_1X32, "32x32": L.LPFA_BLK_32X32}[block]
    q, sf, sf_mma, sf_mma_t, d = L.mx_gemm_quantize(
        _dev(pa), _dev(_gemm_sf_layout(sa)), _dev(pb), _dev(_gemm_sf_layout(sb)), blk,
        with_fp32=True)
    q2, sf2, sf_mma2, sf_mma_t2, _ = L.mx_gemm_quantize(
        _dev(pa), _dev(_gemm_sf_layout(sa)), _dev(pb), _dev(_gemm_sf_layout(sb)), blk)
    torch.cuda.synchronize()
    dk = d.cpu().numpy().astype(np.float64)
    want_d = mx.mx_gemm(pa, sa, pb, sb)
    scale = np.abs(mx.dq_1x32(pa, sa)) @ np.abs(mx.dq_1x32(pb, sb)).T
    assert np.all(np.abs(dk - want_d) <= 1e-5 * scale + 1e-30)
    want = layouts.gemm_quantize(dk, block)
    for got in ((q, sf, sf_mma, sf_mma_t), (q2, sf2, sf_mma2, sf_mma_t2)):
        assert np.array_equal(got[0].cpu().numpy(), want["payload"])
        assert np.array_equal(got[1].cpu().numpy(), want["sf"])
        assert np.array_equal(got[2].cpu().numpy(), want["sf_mma"])
        if block == "32x32":
            assert np.array_equal(got[3].cpu().numpy(), want["sf_mma_t"])


@pytest.mark.parametrize("block", ["1x32", "32x32"])
def test_mx_gemm_quantize_output_feeds_the_next_gemm(L, block):
    """The quantized result, with its tensor-core scale arrangement, as the
    A operand of a second block-scaled GEMM: contraction over N with the rows
    = M arrangement, and (square blocks) contraction over M with the
    transposed payload and the rows = N arrangement."""
    M, N, K, P = 256, 512, 256, 256
    pa, sa, pb, sb = _operands(M, N, K, seed=3)
    blk = {"1x32": L.LPFA_BLK_1X32, "32x32": L.LPFA_BLK_32X32}[block]
    q, sf, sf_mma, sf_mma_t, _ = L.mx_gemm_quantize(
        _dev(pa), _dev(_gemm_sf_layout(sa)), _dev(pb), _dev(_gemm_sf_layout(sb)), blk)
    torch.cuda.synchronize()
    qn, sfn = q.cpu().numpy(), sf.cpu().numpy()
    rows_sc = sfn if block == "1x32" else np.repeat(sfn, 32, axis=0)      # [M, N/32]
    pc, sc = mx.quantize_1x32(np.random.default_rng(5).standard_normal((P, N)))
    e = torch.empty((M, P), dtype=torch.float32, device="cuda")
    L.lpfa_mx_gemm(q, sf_mma, _dev(pc), _dev(_gemm_sf_layout(sc)), e)
    torch.cuda.synchronize()
    want = mx.mx_gemm(qn, rows_sc, pc, sc)
    scale = np.abs(mx.dq_1x32(qn, rows_sc)) @ np.abs(mx.dq_1x32(pc, sc)).T
    assert np.all(np.abs(e.cpu().numpy() - want) <= 1e-5 * scale + 1e-30)
    if block == "32x32":
        pt, st = mx.quantize_1x32(np.random.default_rng(6).standard_normal((P, M)))
        f = torch.empty((N, P), dtype=torch.float32, device="cuda")
        L.lpfa_mx_gemm(_dev(qn.T), sf_mma_t, _dev(pt), _dev(_gemm_sf_layout(st)), f)
        torch.cuda.synchronize()
        cols_sc = np.repeat(sfn.T, 32, axis=0)                            # [N, M/32]
        want_t = mx.mx_gemm(qn.T, cols_sc, pt, st)
        scale_t = np.abs(mx.dq_1x32(qn.T, cols_sc)) @ np.abs(mx.dq_1x32(pt, st)).T
        assert np.all(np.abs(f.cpu().numpy() - want_t) <= 1e-5 * scale_t + 1e-30)


# E4M3 magnitudes (torch's decoder) and the decision boundaries between them:
# the midpoints, and 0 (the sign of a zero code)
_GRID = torch.arange(0, 127, dtype=torch.uint8).view(
    torch.float8_e4m3fn).to(torch.float64).numpy()
_BOUNDS = np.concatenate([[0.0], 0.5 * (_GRID[:-1] + _GRID[1:])])


def _blocks(x, block):
    M, N = x.shape
    if block == "1x32":
        return x.reshape(M, N // 32, 32)
    return x.reshape(M // 32, 32, N // 32, 32).transpose(0, 2, 1, 3).reshape(
        M // 32, N // 32, 1024)


def _open_blocks(exact, bound, block):
    """Blocks whose codes the accumulation bound leaves open: the block
    maximum's binade (the scale) can change within the bound, or some
    element lies within the bound of a rounding boundary at that scale."""
    xb, bb = np.abs(_blocks(exact, block)), _blocks(bound, block)
    amax, bmax = xb.max(-1), bb.max(-1)
    lo = np.floor(np.log2(np.maximum(amax - bmax, 1e-300)))
    hi = np.floor(np.log2(amax + bmax))
    e = np.floor(np.log2(np.maximum(amax, 1e-300))) - 8
    y, dy = xb * 2.0 ** -e[..., None], bb * 2.0 ** -e[..., None]
    i = np.searchsorted(_BOUNDS, y)
    up = _BOUNDS[np.minimum(i, len(_BOUNDS) - 1)]
    down = _BOUNDS[np.maximum(i - 1, 0)]
    near = (np.abs(up - y) <= dy) | (np.abs(y - down) <= dy)
    return (lo != hi) | near.any(-1)


@pytest.mark.parametrize("block", ["1x32", "32x32"])
def test_mx_gemm_quantize_codes_against_exact_product(L, block):
    """The fused codes against the oracle's quantization of the exact fp64
    product.  A block may differ only where the accumulation bound leaves its
    decision open; how many blocks were open and how many differed is
    printed.  Bound: 1e-6 of sum |a||b| at K = 128 (4 fp32 additions of exact
    32-term block products), ten times the largest difference measured on
    this GPU (9.8e-8)."""
    M, N, K = 384, 768, 128
    pa, sa, pb, sb = _operands(M, N, K, seed=77)
    blk = {"1x32": L.LPFA_BLK_1X32, "32x32": L.LPFA_BLK_32X32}[block]
    q, sf, _, _, d = L.mx_gemm_quantize(
        _dev(pa), _dev(_gemm_sf_layout(sa)), _dev(pb), _dev(_gemm_sf_layout(sb)), blk,
        with_fp32=True)
    torch.cuda.synchronize()
    exact = mx.mx_gemm(pa, sa, pb, sb)
    absprod = np.abs(mx.dq_1x32(pa, sa)) @ np.abs(mx.dq_1x32(pb, sb)).T
    bound = 1e-6 * absprod
    # observed accumulation error, for the record (decides nothing)
    print("max |d - exact| / sum|a||b| =",
          float(np.max(np.abs(d.cpu().numpy() - exact) / absprod)))
    want = layouts.gemm_quantize(exact, block)
    got_p, got_s = q.cpu().numpy(), sf.cpu().numpy()
    scale_b = got_s if block == "32x32" else got_s.reshape(M, N // 32)
    want_s = want["sf"] if block == "32x32" else want["sf"].reshape(M, N // 32)
    differ = np.any(_blocks(got_p, block) != _blocks(want["payload"], block), -1) | \
        (scale_b != want_s)
    open_ = _open_blocks(exact, bound, block)
    print(f"{block}: {differ.sum()} of {differ.size} blocks differ, "
          f"{open_.sum()} open")
    assert not np.any(differ & ~open_)
    # the check decides most blocks
    assert open_.mean() < (0.1 if block == "1x32" else 0.6)


# ------------------------------------------------------------ grouped GEMM
def _mx_operand(R, K, seed):
    g = torch.Generator().manual_seed(seed)
    x = (torch.randn(R, K, generator=g) * torch.exp(torch.randn(R, 1, generator=g))).bfloat16()
    p, s = mx.quantize_1x32(x.float().numpy().astype(np.float64))
    dev = lambda z: torch.from_numpy(np.ascontiguousarray(z)).cuda()
    return dev(p), dev(_gemm_sf_layout(s)), p, s


def test_mx_gemm_grouped_equals_separate(L):
    """Two problems in one launch (a short-contraction one with a ragged M and
    many tiles, a long-contraction one with few) give bit-for-bit the results
    of separate launches, which match the oracle."""
    shapes = [(1284, 512, 256), (256, 768, 1408)]
    ops = []
    for i, (M, N, K) in enumerate(shapes):
        a, sa, pa, qa = _mx_operand(M, K, 10 + i)
        b, sb, pb, qb = _mx_operand(N, K, 20 + i)
        ops.append((a, sa, b, sb, M, N, pa, qa, pb, qb))
    sep = []
    for a, sa, b, sb, M, N, *_ in ops:
        d = torch.empty((M, N), dtype=torch.float32, device="cuda")
        L.lpfa_mx_gemm(a, sa, b, sb, d)
        sep.append(d)
    grp = [torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
           for _, _, _, _, M, N, *_ in ops]
    L.lpfa_mx_gemm_grouped([(a, sa, b, sb, d) for (a, sa, b, sb, *_), d in zip(ops, grp)])
    one = torch.full_like(sep[0], float("nan"))
    L.lpfa_mx_gemm_grouped([(ops[0][0], ops[0][1], ops[0][2], ops[0][3], one)])
    torch.cuda.synchronize()
    for d, e in zip(grp, sep):
        assert torch.equal(d, e)
    assert torch.equal(one, sep[0])
    for (a, sa, b, sb, M, N, pa, qa, pb, qb), d in zip(ops, sep):
        want = mx.mx_gemm(pa, qa, pb, qb)
        bound = 1e-5 * (np.abs(mx.dq_1x32(pa, qa)) @ np.abs(mx.dq_1x32(pb, qb)).T)
        assert np.all(np.abs(d.cpu().numpy().astype(np.float64) - want) <= bound + 1e-30)


def test_mx_gemm_grouped_rejects_bad_arguments(L):
    arr = (L.lpfa_gemm_problem * 3)()
    assert L._mx_gemm_grouped(arr, 3, None) == L.LPFA_ERR_INVALID_ARG
    assert L._mx_gemm_grouped(arr, 0, None) == L.LPFA_ERR_INVALID_ARG
    assert L._mx_gemm_grouped(arr, 1, None) == L.LPFA_ERR_INVALID_ARG   # null pointers
