"""Pins for the oracle's attention (CPU only).

The exact oracle is checked against torch's own fp64 scaled-dot-product
attention and autograd (independent library routines) and against central
finite differences; the MXFP8 oracle is checked, with quantization switched
off, against the same library routines for several key-tile sizes and
rescaling thresholds (the online-softmax bookkeeping must not change the
result), and with quantization on against closed forms (Q = 0 gives uniform
attention: O is the mean of the quantized V and LSE = ln(#keys)) and the
error bound against exact attention.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import workloads
from oracle import attention as A
from oracle import mx


def _sdpa_with_grads(q, k, v, do, causal, scale):
    qt = torch.from_numpy(q).clone().requires_grad_(True)
    kt = torch.from_numpy(k).clone().requires_grad_(True)
    vt = torch.from_numpy(v).clone().requires_grad_(True)
    hq, hkv = q.shape[1], k.shape[1]
    kk = kt.permute(1, 0, 2)[None].repeat_interleave(hq // hkv, dim=1)
    vv = vt.permute(1, 0, 2)[None].repeat_interleave(hq // hkv, dim=1)
    o = F.scaled_dot_product_attention(qt.permute(1, 0, 2)[None], kk, vv,
                                       is_causal=causal, scale=scale)
    o = o[0].permute(1, 0, 2)
    o.backward(torch.from_numpy(do))
    lse = torch.logsumexp(
        scale * torch.einsum("qhd,khd->hqk", qt.detach(),
                             kt.detach().repeat_interleave(hq // hkv, dim=1))
        + (torch.triu(torch.full((q.shape[0], q.shape[0]), -math.inf,
                                 dtype=torch.float64), 1) if causal else 0),
        dim=-1)
    return (o.detach().numpy(), lse.numpy(), qt.grad.numpy(),
            kt.grad.numpy(), vt.grad.numpy())


def _rand(rng, L, hq, hkv, d):
    return (rng.standard_normal((L, hq, d)), rng.standard_normal((L, hkv, d)),
            rng.standard_normal((L, hkv, d)), rng.standard_normal((L, hq, d)))


def _relfro(a, b):
    return np.linalg.norm(a - b) / np.linalg.norm(b)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("hq,hkv", [(2, 2), (4, 2)])
def test_exact_matches_torch_sdpa_and_autograd(rng, causal, hq, hkv):
    L, d = 70, 32
    q, k, v, do = _rand(rng, L, hq, hkv, d)
    scale = 1 / math.sqrt(d)
    o, lse, dq, dk, dv = _sdpa_with_grads(q, k, v, do, causal, scale)
    res = A.exact_attention(q, k, v, causal=causal, softmax_scale=scale,
                            cu_seqlens=[0, L], do=do)
    assert np.allclose(res["o"], o, rtol=1e-12, atol=1e-12)
    assert np.allclose(res["lse"], lse, rtol=1e-12, atol=1e-12)
    for got, want in ((res["dq"], dq), (res["dk"], dk), (res["dv"], dv)):
        assert np.allclose(got, want, rtol=1e-10, atol=1e-12)


def test_exact_bwd_finite_difference(rng):
    """Central differences of <dO, O> w.r.t. Q, K, V (h = 1e-6)."""
    L, d = 12, 8
    q, k, v, do = _rand(rng, L, 1, 1, d)
    scale = 0.7
    res = A.exact_attention(q, k, v, causal=True, softmax_scale=scale,
                            cu_seqlens=[0, L], do=do)
    h = 1e-6

    def f(qq, kk, vv):
        o = A.exact_attention(qq, kk, vv, causal=True, softmax_scale=scale,
                              cu_seqlens=[0, L])["o"]
        return float((o * do).sum())

    for name, x, g in (("q", q, res["dq"]), ("k", k, res["dk"]),
                       ("v", v, res["dv"])):
        num = np.zeros_like(x)
        for idx in np.ndindex(*x.shape):
            xp = x.copy(); xp[idx] += h
            xm = x.copy(); xm[idx] -= h
            args = {"q": q, "k": k, "v": v}
            args[name] = xp; fp = f(args["q"], args["k"], args["v"])
            args[name] = xm; fm = f(args["q"], args["k"], args["v"])
            num[idx] = (fp - fm) / (2 * h)
        assert np.linalg.norm(num - g) / np.linalg.norm(g) < 1e-6, name


def test_softmax_rows_sum_to_one(rng):
    """With V = 1 every output row is sum_j P_ij / l_i = 1."""
    L, d = 50, 16
    q, k, _, _ = _rand(rng, L, 2, 2, d)
    v = np.ones((L, 2, d))
    for causal in (False, True):
        o = A.exact_attention(q, k, v, causal=causal, softmax_scale=0.3,
                              cu_seqlens=[0, L])["o"]
        assert np.abs(o - 1).max() < 1e-15
        o2 = A.mx_attention_fwd(q, k, v, causal=causal, softmax_scale=0.3,
                                cu_seqlens=[0, L], quantize=False,
                                kv_tile=16)["o"]
        assert np.abs(o2 - 1).max() < 1e-14


@pytest.mark.parametrize("kv_tile,tau", [(128, 8.0), (16, 0.0), (32, 8.0),
                                         (16, 2.0), (1000, 0.0)])
@pytest.mark.parametrize("causal", [False, True])
def test_online_unquantized_equals_exact(rng, kv_tile, tau, causal):
    """The blockwise online softmax (any tile, any rescale threshold) with
    quantization off equals torch SDPA; varlen and GQA included."""
    cu = np.array([0, 37, 137, 300])
    T, d = cu[-1], 32
    q, k, v, _ = _rand(rng, T, 4, 2, d)
    q *= 3  # spread logits so the reference max moves
    scale = 1 / math.sqrt(d)
    res = A.mx_attention_fwd(q, k, v, causal=causal, softmax_scale=scale,
                             cu_seqlens=cu, kv_tile=kv_tile,
                             rescale_threshold=tau, quantize=False)
    for s in range(3):
        a, b = cu[s], cu[s + 1]
        o, lse, *_ = _sdpa_with_grads(q[a:b], k[a:b], v[a:b],
                                      np.zeros_like(q[a:b]), causal, scale)
        assert np.allclose(res["o"][a:b], o, rtol=1e-11, atol=1e-12)
        assert np.allclose(res["lse"][:, a:b], lse, rtol=1e-11, atol=1e-12)


def test_q_zero_gives_mean_of_quantized_v(rng):
    """Q = 0: every logit is 0, P = 1 exactly (quantized P = 1 too), so O is
    the mean of the quantized V over the visible keys and LSE = ln(#keys)."""
    L, d = 200, 64
    q = np.zeros((L, 2, d)); k = rng.standard_normal((L, 2, d))
    v = rng.standard_normal((L, 2, d))
    for causal in (False, True):
        res = A.mx_attention_fwd(q, k, v, causal=causal, softmax_scale=0.125,
                                 cu_seqlens=[0, L])
        vq = mx.fake_quant_rows(v)
        n = np.arange(1, L + 1) if causal else np.full(L, L)
        mean = (np.cumsum(vq, 0) / n[:, None, None]) if causal else \
            np.broadcast_to(vq.mean(0), vq.shape)
        assert np.allclose(res["o"], mean, rtol=1e-13, atol=1e-13)
        assert np.allclose(res["lse"], np.log(n)[None, :], rtol=1e-14)


def test_quantized_fwd_within_bound_of_exact():
    """O within 8e-2 relative Frobenius of fp64 unquantized attention on the
    tiny and (one head of the) outlier workloads."""
    w = workloads.get_config("tiny")
    x = workloads.make_inputs(w)
    mxr = A.mx_attention_fwd(x["q"], x["k"], x["v"], causal=w.causal,
                             softmax_scale=w.softmax_scale)
    ex = A.exact_attention(x["q"], x["k"], x["v"], causal=w.causal,
                           softmax_scale=w.softmax_scale)
    err = _relfro(mxr["o"], ex["o"])
    assert err < 8e-2
    assert err > 1e-3           # quantization really happened
    assert np.abs(mxr["lse"] - ex["lse"]).max() < 5e-2


def test_quantized_gemm_operands_are_the_pages_quantization_points(rng):
    """The forward's quantized Q/K/V equal the codec's 1x32 (head_dim) and
    32-key quantizers (pins which axis each operand is blocked along)."""
    cu = np.array([0, 40, 100])
    q, k, v, _ = _rand(rng, 100, 2, 2, 64)
    qd, kd, vd = A.quantize_fwd_operands(q, k, v, cu)
    assert np.array_equal(qd, mx.dq_1x32(*mx.quantize_1x32(q)))
    assert np.array_equal(vd[40:], mx.dq_rows(*mx.quantize_along_rows(v[40:])))
    # a 32-key block of V shares one scale per channel
    sc = mx.quantize_along_rows(v[:40])[1]
    assert sc.shape == (2, 2, 64)


@pytest.mark.parametrize("causal", [False, True])
def test_bwd_unquantized_matches_autograd(rng, causal):
    """Backward with quantization off equals autograd (dQ within FP16
    accumulation error), GQA and varlen included."""
    cu = np.array([0, 64, 160])
    T, d = cu[-1], 32
    q, k, v, do = _rand(rng, T, 4, 2, d)
    scale = 1 / math.sqrt(d)
    ex = A.exact_attention(q, k, v, causal=causal, softmax_scale=scale,
                           cu_seqlens=cu, do=do)
    res = A.mx_attention_bwd(q, k, v, ex["o"], do, ex["lse"], causal=causal,
                             softmax_scale=scale, cu_seqlens=cu,
                             quantize=False, kv_tile=32)
    for s in range(2):
        a, b = cu[s], cu[s + 1]
        _, _, dq, dk, dv = _sdpa_with_grads(q[a:b], k[a:b], v[a:b], do[a:b],
                                            causal, scale)
        assert np.allclose(res["dk"][a:b], dk, rtol=1e-10, atol=1e-12)
        assert np.allclose(res["dv"][a:b], dv, rtol=1e-10, atol=1e-12)
        assert _relfro(res["dq"][a:b], dq) < 2e-3     # fp16 accumulation


def test_bwd_dq_static_scale(rng):
    """A power-of-two static scale changes dQ only through fp16 rounding of
    tiny values; a scale that pushes dQ into fp16 subnormals visibly hurts."""
    cu = np.array([0, 96])
    q, k, v, do = _rand(rng, 96, 1, 1, 32)
    ex = A.exact_attention(q, k, v, causal=True, softmax_scale=0.2,
                           cu_seqlens=cu, do=do)
    kw = dict(causal=True, softmax_scale=0.2, cu_seqlens=cu, kv_tile=32,
              quantize=False)
    r1 = A.mx_attention_bwd(q, k, v, ex["o"], do, ex["lse"], **kw)
    r4 = A.mx_attention_bwd(q, k, v, ex["o"], do, ex["lse"],
                            dq_static_scale=4.0, **kw)
    tiny = A.mx_attention_bwd(q, k, v, ex["o"], do, ex["lse"],
                              dq_static_scale=2.0 ** -20, **kw)
    assert _relfro(r4["dq"], ex["dq"]) < 2e-3
    assert _relfro(r1["dq"], ex["dq"]) < 2e-3
    assert _relfro(tiny["dq"], ex["dq"]) > 1e-2
    assert np.array_equal(r1["dk"], r4["dk"])


def test_bwd_quantized_close_to_exact_and_sampling_consistent(rng):
    """Quantized gradients stay near exact ones; computing a sample of rows
    gives the same numbers as the full computation."""
    w = workloads.get_config("tiny")
    x = workloads.make_inputs(w)
    ex = A.exact_attention(x["q"], x["k"], x["v"], causal=False,
                           softmax_scale=w.softmax_scale, do=x["do"])
    fw = A.mx_attention_fwd(x["q"], x["k"], x["v"], causal=False,
                            softmax_scale=w.softmax_scale)
    o16 = torch.from_numpy(fw["o"]).to(torch.bfloat16)
    full = A.mx_attention_bwd(x["q"], x["k"], x["v"], o16, x["do"],
                              fw["lse"], causal=False,
                              softmax_scale=w.softmax_scale)
    for g in ("dq", "dk", "dv"):
        assert _relfro(full[g], ex[g]) < 0.15, g
    rows = np.arange(64, 128)
    part = A.mx_attention_bwd(x["q"], x["k"], x["v"], o16, x["do"],
                              fw["lse"], causal=False,
                              softmax_scale=w.softmax_scale, q_rows=rows,
                              k_rows=rows)
    for g in ("dq", "dk", "dv"):
        assert np.array_equal(part[g][:, 64:128], full[g][:, 64:128]), g
        assert np.all(np.isnan(part[g][:, :64]))


def test_bwd_causal_sampling_consistent(rng):
    cu = np.array([0, 200])
    q, k, v, do = _rand(rng, 200, 2, 1, 32)
    fw = A.mx_attention_fwd(q, k, v, causal=True, softmax_scale=0.3,
                            cu_seqlens=cu)
    full = A.mx_attention_bwd(q, k, v, fw["o"], do, fw["lse"], causal=True,
                              softmax_scale=0.3, cu_seqlens=cu)
    part = A.mx_attention_bwd(q, k, v, fw["o"], do, fw["lse"], causal=True,
                              softmax_scale=0.3, cu_seqlens=cu,
                              q_rows=np.arange(160, 200),
                              k_rows=np.arange(96, 128))
    assert np.array_equal(part["dq"][160:200], full["dq"][160:200])
    assert np.array_equal(part["dk"][96:128], full["dk"][96:128])
    assert np.array_equal(part["dv"][96:128], full["dv"][96:128])


@pytest.mark.parametrize("causal", [False, True])
def test_exact_chunked_equals_whole_head(rng, causal):
    """Query-row blocks (one ragged) give the whole-head result."""
    L, d = 150, 16
    q, k, v, _ = _rand(rng, L, 1, 1, d)
    o, lse = A.exact_fwd_head(q[:, 0], k[:, 0], v[:, 0], causal, 0.4)
    oc, lc = A.exact_fwd_head_chunked(q[:, 0], k[:, 0], v[:, 0], causal, 0.4,
                                      chunk=64)
    assert np.allclose(oc, o, rtol=1e-13, atol=1e-14)
    assert np.allclose(lc, lse, rtol=1e-14, atol=1e-14)
