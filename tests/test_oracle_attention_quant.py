"""Pins for the quantization points inside the attention oracle (CPU only).

Each test fixes one step that the looser error bounds cannot see:

* the forward's P_hat: a hand-worked 64-key example (the fixture in
  tests/golden/fwd_p_quantization_example.txt), under three key-tile readings;
  and a restatement on random inputs with one key tile and no selective
  rescaling, where P_hat is the 1x32 block rounding of 2^(x - rowmax);
* the backward's operands: Q, K, dO in 32x32 blocks over (token, head_dim)
  per head, V in 1x32 blocks along head_dim;
* the backward's P_tilde and dS_tilde: with Q = I and dO = I the oracle's dV
  is P_tilde^T and its dK is c * dS_tilde^T, so both can be read off and
  compared with 32x32 block roundings of P and dS computed here.

The block roundings below are written independently of ``oracle.mx``: scales
from ``math.frexp`` of each block's maximum, elements by brute-force nearest
search over torch's own E4M3 decode of all codes (ties to the even code,
saturation at 448).  Sources: "Low Precision Flash Attention 4 ...",
paragraphs 2-3; "Low-Precision FlashAttention-4 ...", "Understanding OCP
MXFP8 Microscaling on Blackwell".
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import attention as A

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

# non-negative finite E4M3 magnitudes, codes 0..126 (torch's decoder)
_GRID = torch.arange(0, 127, dtype=torch.uint8).view(
    torch.float8_e4m3fn).to(torch.float64).numpy()
_EVEN = (np.arange(127) % 2) == 0


def _round_e4m3(a):
    """Nearest E4M3 value of each element of ``a`` (fp64), by exhaustive
    search: ties go to the even code, magnitudes above 448 saturate."""
    a = np.asarray(a, np.float64)
    mag = np.minimum(np.abs(a), 448.0)
    d = np.abs(mag[..., None] - _GRID)
    cand = d == d.min(axis=-1, keepdims=True)
    even = cand & _EVEN
    pick = np.where(even.any(-1), even.argmax(-1), cand.argmax(-1))
    return np.sign(a) * _GRID[pick]


def _round_block(blk):
    """One MX block (any shape) rounded with one shared scale 2^e,
    e = floor(log2 amax) - 8."""
    amax = float(np.abs(blk).max())
    if amax == 0.0:
        return np.zeros_like(blk)
    e = math.frexp(amax)[1] - 1 - 8
    return _round_e4m3(blk * 2.0 ** -e) * 2.0 ** e


def _blocks_1x32(x):
    """1x32 blocks along the last axis (length a multiple of 32)."""
    out = np.empty_like(x)
    for idx in np.ndindex(*x.shape[:-1]):
        for c in range(0, x.shape[-1], 32):
            out[idx + (slice(c, c + 32),)] = _round_block(x[idx + (slice(c, c + 32),)])
    return out


def _blocks_32x32(x):
    """32x32 blocks over a 2-D array; rows and columns multiples of 32."""
    out = np.empty_like(x)
    for r in range(0, x.shape[0], 32):
        for c in range(0, x.shape[1], 32):
            out[r:r + 32, c:c + 32] = _round_block(x[r:r + 32, c:c + 32])
    return out


def _blocks_32_rows(x):
    """Blocks of 32 consecutive rows per column (x: [L, D], L % 32 == 0)."""
    return _blocks_1x32(x.T).T


# ------------------------------------------------------------ forward P_hat
def _golden_rows():
    rows = []
    with open(os.path.join(GOLDEN, "fwd_p_quantization_example.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            key, x, *phat = line.split()
            rows.append((int(key), float(x), [float(Fraction(p)) for p in phat]))
    return rows


@pytest.mark.parametrize("reading,kv_tile,tau", [("onetile", 64, 8.0),
                                                 ("tau8", 32, 8.0),
                                                 ("tau0", 32, 0.0)])
def test_fwd_p_hat_hand_worked(reading, kv_tile, tau):
    rows = _golden_rows()
    col = {"onetile": 0, "tau8": 1, "tau0": 2}[reading]
    x = np.array([r[1] for r in rows])
    p_hat = np.array([r[2][col] for r in rows])
    L, D = 64, 32
    q = np.zeros((1, 1, D)); q[0, 0, 0] = 1.0
    k = np.zeros((L, 1, D)); k[:, 0, 0] = x
    v = np.zeros((L, 1, D)); v[np.arange(L), 0, np.arange(L) % 32] = 1.0
    # query row 0 of a one-row "sequence" would see one key under causal
    # masking; the example is non-causal, with the query placed at row 0 of
    # 64 (the other 63 query rows are zero and not compared)
    qq = np.zeros((L, 1, D)); qq[0] = q[0]
    res = A.mx_attention_fwd(qq, k, v, causal=False, softmax_scale=math.log(2),
                             cu_seqlens=[0, L], kv_tile=kv_tile,
                             rescale_threshold=tau)
    # weights and running sum as the hand-worked readings define them
    p = 2.0 ** x
    if reading == "onetile":
        w, l = p_hat, (p / 2 ** 0.5).sum()
    elif reading == "tau8":
        w, l = p_hat, p.sum()
    else:
        alpha = 2 ** -0.5
        w = np.concatenate([alpha * p_hat[:32], p_hat[32:]])
        l = alpha * p[:32].sum() + (p[32:] / 2 ** 0.5).sum()
    want = (w[:32] + w[32:]) / l
    assert np.allclose(res["o"][0, 0], want, rtol=1e-14, atol=0)
    assert abs(res["lse"][0, 0] - math.log(p.sum())) < 1e-14


def test_fwd_p_hat_restated_one_tile(rng):
    """With one key tile and threshold 0 the reference max is the row max, so
    O = (P_hat V_hat) / l with P_hat = 1x32 block rounding of 2^(x - rowmax)
    along keys, l the sum of the unrounded P, Q_hat and K_hat 1x32 along
    head_dim and V_hat in 32-key blocks per channel."""
    L, D, c = 96, 64, 0.125
    q = 2.0 * rng.standard_normal((L, 1, D))
    k = rng.standard_normal((L, 1, D))
    v = rng.standard_normal((L, 1, D))
    for causal in (False, True):
        res = A.mx_attention_fwd(q, k, v, causal=causal, softmax_scale=c,
                                 cu_seqlens=[0, L], kv_tile=L,
                                 rescale_threshold=0.0)
        qh, kh = _blocks_1x32(q[:, 0]), _blocks_1x32(k[:, 0])
        vh = _blocks_32_rows(v[:, 0])
        x = (c / math.log(2)) * (qh @ kh.T)
        if causal:
            x = np.where(np.triu(np.ones((L, L), bool), 1), -np.inf, x)
        p = np.exp2(x - x.max(axis=1, keepdims=True))
        p_hat = _blocks_1x32(p)
        o = (p_hat @ vh) / p.sum(axis=1, keepdims=True)
        assert np.allclose(res["o"][:, 0], o, rtol=1e-11, atol=1e-13)
        # and P_hat really differs from P (the pin would be vacuous otherwise)
        assert np.abs(p_hat - p).max() > 1e-3


# ----------------------------------------------------- backward operands
def test_bwd_operands_square_per_head_and_v_along_head_dim(rng):
    cu = np.array([0, 64, 160])
    T, H, D = 160, 2, 64
    q, k, v, do = (rng.standard_normal((T, H, D)) * s
                   for s in (1.0, 3.0, 1.0, 0.5))
    # one outlier channel makes 1x32 and 32x32 blocks disagree
    q[:, :, 5] *= 40.0
    qd, kd, vd, dod = A.quantize_bwd_operands(q, k, v, do, cu)
    for name, x, got in (("q", q, qd), ("k", k, kd), ("do", do, dod)):
        for s in range(2):
            a, b = cu[s], cu[s + 1]
            for h in range(H):
                want = _blocks_32x32(x[a:b, h])
                assert np.array_equal(got[a:b, h], want), (name, s, h)
    assert np.array_equal(vd.reshape(T * H, D), _blocks_1x32(v.reshape(T * H, D)))


# ------------------------------------------- backward P_tilde and dS_tilde
def test_bwd_p_and_ds_square_blocks_read_off_dv_dk(rng):
    """Q = I and dO = I (both exact under 32x32 blocks) give
    dV = P_tilde^T dO_tilde = P_tilde^T and dK = c dS_tilde^T Q_tilde =
    c dS_tilde^T, so the oracle's quantized P and dS are visible in its
    outputs.  They must be the 32x32 (query, key) block roundings of
    P = exp(c S - LSE) and dS = P (dP - D) computed from the quantized
    operands; dQ = c dS_tilde K_tilde rounded to FP16 (one 64-key tile)."""
    L = D = 64
    c = 0.3
    q = np.eye(L)[:, None, :]
    do = np.eye(L)[:, None, :]
    k = 3.0 * rng.standard_normal((L, 1, D))
    v = rng.standard_normal((L, 1, D))
    o = torch.from_numpy(rng.standard_normal((L, 1, D))).to(torch.bfloat16)
    o64 = o.double().numpy()
    kt = _blocks_32x32(k[:, 0])
    vt = _blocks_1x32(v[:, 0])
    s = c * kt.T                                # S = c Q_tilde K_tilde^T
    lse = np.log(np.exp(s).sum(axis=1))
    res = A.mx_attention_bwd(q, k, v, o, do, lse[None, :], causal=False,
                             softmax_scale=c, cu_seqlens=[0, L])
    p = np.exp(s - lse[:, None])
    dp = vt.T                                   # dO_tilde V_tilde^T
    delta = np.diag(o64[:, 0])                  # D_i = sum_d dO_id O_id
    ds = p * (dp - delta[:, None])
    p_t, ds_t = _blocks_32x32(p), _blocks_32x32(ds)
    assert np.allclose(res["dv"][:, 0], p_t.T, rtol=1e-13, atol=0)
    assert np.allclose(res["dk"][:, 0], c * ds_t.T, rtol=1e-13, atol=1e-300)
    dq = c * ds_t @ kt
    assert np.all(np.abs(res["dq"][:, 0] - dq) <= 2.0 ** -11 * np.abs(dq) + 1e-7)
    # the pin is not vacuous: rounding moved both
    assert np.abs(p_t - p).max() > 1e-4 and np.abs(ds_t - ds).max() > 1e-4


# ------------------------------------------------------- key-tile reading
def test_product_key_tiles_equal_the_oracle_readings():
    """The forward kernel's online softmax walks keys in tiles of the length
    the oracle's reading fixes (the rounding of P moves with the tile's
    reference max), and the backward adds FP16 dQ partials per key tile of
    the oracle's backward tile."""
    import mxfp8_block_scaled_quantizer_gb300 as pkg
    assert pkg.FWD_KV_TILE == A.FWD_KEY_TILE
    assert pkg.BWD_KV_TILE == A.BWD_KEY_TILE
