"""Pins for the oracle of the fused RMSNorm + MX quantizer (CPU only).

The fp32 sequence (``norm.rmsnorm_fp32``) is tied to the fp64 definition and
to torch's own rms_norm, to closed forms (constant and zero rows, exact
integer sums, fp32 overflow), and the quantized output to the E4M3 error
bound around the fp64 RMSNorm.  The operation is the fused producer of "Low
Precision Flash Attention 4: End-to-End Block-Scaled Attention for
Blackwell", paragraph 2.
"""
import math

import numpy as np
import pytest
import torch

from oracle import mx, norm


def _bf16(a):
    return torch.tensor(np.asarray(a, dtype=np.float32)).bfloat16().float().numpy()


@pytest.mark.parametrize("n,eps", [(256, 1e-6), (4096, 1e-5), (512, 0.5)])
def test_fp32_sequence_within_rounding_of_fp64(n, eps, rng):
    x = _bf16(rng.standard_normal((6, n)) * np.exp(rng.standard_normal((6, 1))))
    w = _bf16(rng.standard_normal(n))
    y, rstd = norm.rmsnorm_fp32(x, w, eps)
    y64 = norm.rmsnorm_fp64(x, w, eps)
    r64 = 1.0 / np.sqrt(np.mean(x.astype(np.float64) ** 2, axis=1) + eps)
    # fp32 sum of n terms, 4 correctly rounded steps, two products
    tol = (n / 32 + 5 + 4) * 2.0 ** -24
    assert np.all(np.abs(rstd - r64) <= tol * r64)
    nz = np.abs(y64) > 0
    assert np.all(np.abs(y[nz] - y64[nz]) <= (tol + 2 * 2.0 ** -24) * np.abs(y64[nz]))


def test_fp64_definition_matches_torch_rms_norm(rng):
    x = rng.standard_normal((4, 384))
    w = rng.standard_normal(384)
    ref = torch.nn.functional.rms_norm(torch.tensor(x), (384,), torch.tensor(w), eps=1e-5)
    assert np.allclose(norm.rmsnorm_fp64(x, w, 1e-5), ref.numpy(), rtol=1e-12, atol=0)


def test_constant_and_zero_rows():
    n, eps = 128, 2.0 ** -20
    x = np.zeros((3, n), dtype=np.float32)
    x[0] = 3.0
    x[1] = -0.5
    w = np.full(n, 2.0, dtype=np.float32)
    y, rstd = norm.rmsnorm_fp32(x, w, eps)
    for t, c in ((0, 3.0), (1, -0.5)):
        want = c / math.sqrt(c * c + eps) * 2.0
        assert np.allclose(y[t], want, rtol=2 ** -22, atol=0)
    assert np.all(y[2] == 0) and rstd[2] == np.float32(1.0 / np.sqrt(np.float32(eps)))


def test_integer_rows_sum_exactly():
    # squares of small integers: every partial sum is exact in any order, so
    # the fixed-order fp32 sum equals the exact sum
    rng = np.random.default_rng(7)
    for n in (64, 1024, 4096):
        row = rng.integers(-40, 41, size=n).astype(np.float32)
        assert float(norm._sum_squares_fp32(row)) == math.fsum(float(v) ** 2 for v in row)


def test_fp32_overflow_gives_zero_output():
    # x^2 beyond fp32 range: ss = inf, rstd = 0, y = 0 (the fp32 sequence)
    n = 64
    x = np.ones((1, n), dtype=np.float32)
    x[0, 5] = 2.0 ** 70
    y, rstd = norm.rmsnorm_fp32(x, np.ones(n, dtype=np.float32), 1e-6)
    assert rstd[0] == 0.0 and np.all(y == 0)


@pytest.mark.parametrize("block", ["1x32", "32x32"])
def test_quantized_output_within_e4m3_bound(block, rng):
    T, H, D = 64, 4, 32 * 4
    n = H * D
    x = _bf16(rng.standard_normal((T, n)))
    x[3, :64] *= 50.0                                  # a row with outliers
    w = _bf16(1.0 + 0.1 * rng.standard_normal(n))
    out = norm.rms_quantize(x, w, 1e-6, H, np.array([0, T]), block)
    y64 = norm.rmsnorm_fp64(x, w, 1e-6).reshape(T, H, D)
    vals = mx.E4M3_TABLE[out["payload"]]
    if block == "1x32":
        sc = np.repeat(out["sf"].astype(np.int64), 32, axis=2)
    else:
        sc = np.repeat(np.repeat(out["sf"].astype(np.int64), 32, axis=0)[:T], 32, axis=2)
    e = sc - 127
    deq = vals * np.exp2(e)
    # nearest-even rounding: half a step of E4M3 (2^-4 relative for normals,
    # 2^-10 * 2^e absolute in the subnormal range); magnitudes above 448 * 2^e
    # (the scale rule admits block maxima up to 511 * 2^e) saturate to 448;
    # plus fp32 slack
    sat = np.maximum(np.abs(y64) - 448.0 * np.exp2(e), 0.0)
    bound = np.maximum(np.maximum(np.abs(y64) * 2.0 ** -4, np.exp2(e - 10.0)), sat) * (1 + 2.0 ** -18)
    assert np.all(np.abs(deq - y64) <= bound + 1e-6 * np.abs(y64))
    assert np.all(np.sign(deq) * np.sign(y64) >= 0)
    assert out["rstd"].shape == (T,)
