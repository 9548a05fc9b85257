"""Forward parity on the GPU against the quantization-matched oracle (O
relative Frobenius <= 2e-2, LSE absolute <= 1e-3) and against exact fp64
attention (O <= 8e-2 on the i.i.d. workloads), full for small workloads and
sampled (heads, query rows, sequences) at full size in the launch
configuration the bench times."""
import math

import numpy as np
import pytest
import torch

import workloads
from oracle import attention as A

pytestmark = pytest.mark.gpu

TOL_O, TOL_LSE, TOL_EXACT = 2e-2, 1e-3, 8e-2


@pytest.fixture(scope="module")
def L():
    from mxfp8_block_scaled_quantizer_gb300 import build
    build()
    from mxfp8_block_scaled_quantizer_gb300 import lpfa
    return lpfa


def relfro(a, b):
    a = np.asarray(a, np.float64); b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def _run(L, x, w, tau=8.0):
    cu = x["cu_seqlens"] if w.varlen else None
    o, lse = L.mx_attention_forward(x["q"].cuda(), x["k"].cuda(),
                                    x["v"].cuda(), causal=w.causal,
                                    softmax_scale=w.softmax_scale,
                                    cu_seqlens=cu, rescale_threshold=tau)
    torch.cuda.synchronize()
    return o.float().cpu().numpy(), lse.cpu().numpy()


def _tok(a):
    """BSHD -> token-major view."""
    return a.reshape(-1, *a.shape[2:]) if a.ndim == 4 else a


def test_fwd_tiny_full(L):
    w = workloads.get_config("tiny")
    x = workloads.make_inputs(w)
    o, lse = _run(L, x, w)
    ref = A.mx_attention_fwd(x["q"], x["k"], x["v"], causal=w.causal,
                             softmax_scale=w.softmax_scale, kv_tile=A.FWD_KEY_TILE)
    assert relfro(o, ref["o"]) <= TOL_O
    assert np.abs(lse - ref["lse"]).max() <= TOL_LSE
    ex = A.exact_attention(x["q"], x["k"], x["v"], causal=w.causal,
                           softmax_scale=w.softmax_scale)
    assert relfro(o, ex["o"]) <= TOL_EXACT


def test_fwd_outlier_sampled_heads(L):
    w = workloads.get_config("outlier")
    x = workloads.make_inputs(w)
    o, lse = _run(L, x, w)
    heads = [0, 9, 15]
    ref = A.mx_attention_fwd(x["q"], x["k"], x["v"], causal=True,
                             softmax_scale=w.softmax_scale, heads=heads, kv_tile=A.FWD_KEY_TILE)
    for h in heads:
        assert relfro(o[:, :, h], ref["o"][:, :, h]) <= TOL_O, h
        assert np.abs(lse[h] - ref["lse"][h]).max() <= TOL_LSE, h


@pytest.mark.parametrize("name", ["llm", "gqa_long"])
def test_fwd_full_size_sampled(L, name):
    """Full-size launch; oracle on first/last heads and three query tiles
    (first, middle, last) of the first and last sequence."""
    w = workloads.get_config(name)
    x = workloads.make_inputs(w, with_grad_out=False)
    o, lse = _run(L, x, w)
    S = w.seqlen
    rows = np.concatenate([np.arange(0, 128), np.arange(S // 2, S // 2 + 128),
                           np.arange(S - 128, S)])
    heads = [0, w.heads_q - 1]
    ref = A.mx_attention_fwd(x["q"], x["k"], x["v"], causal=w.causal,
                             softmax_scale=w.softmax_scale, heads=heads,
                             seqs=[0, w.batch - 1], rows=rows, kv_tile=A.FWD_KEY_TILE)
    ot = _tok(o); rt = _tok(ref["o"])
    for b in (0, w.batch - 1):
        for h in heads:
            idx = b * S + rows
            assert relfro(ot[idx, h], rt[idx, h]) <= TOL_O, (b, h)
            assert np.abs(lse[h, idx] - ref["lse"][h, idx]).max() <= TOL_LSE
    if name == "llm":   # i.i.d. inputs: also close to exact attention
        q = x["q"][0, :, 0:1]; k = x["k"][0, :, 0:1]; v = x["v"][0, :, 0:1]
        qq = q[S - 128:]
        # exact rows S-128..S-1 see every key
        s = (qq.double()[:, 0] @ k.double()[:, 0].T) * w.softmax_scale
        mask = torch.arange(S)[None, :] > torch.arange(S - 128, S)[:, None]
        s[mask] = -math.inf
        ex = torch.softmax(s, -1) @ v.double()[:, 0]
        assert relfro(o[0, S - 128:, 0], ex.numpy()) <= TOL_EXACT


def test_fwd_varlen_sampled_sequences(L):
    w = workloads.get_config("varlen")
    x = workloads.make_inputs(w, with_grad_out=False)
    o, lse = _run(L, x, w)
    lens = x["lengths"].numpy()
    seqs = sorted({int(lens.argmin()), int(lens.argmax()), 5, 40})
    heads = [0, 15]
    ref = A.mx_attention_fwd(x["q"], x["k"], x["v"], causal=False,
                             softmax_scale=w.softmax_scale,
                             cu_seqlens=x["cu_seqlens"].numpy(), heads=heads,
                             seqs=seqs, kv_tile=A.FWD_KEY_TILE)
    cu = x["cu_seqlens"].numpy()
    for s in seqs:
        a, b = cu[s], cu[s + 1]
        for h in heads:
            assert relfro(o[a:b, h], ref["o"][a:b, h]) <= TOL_O, (s, h)
            assert np.abs(lse[h, a:b] - ref["lse"][h, a:b]).max() <= TOL_LSE


@pytest.mark.parametrize("case", [
    dict(batch=2, seqlen=200, heads_q=4, heads_kv=1, head_dim=128, causal=True),
    dict(batch=1, seqlen=384, heads_q=2, heads_kv=2, head_dim=64, causal=True),
    dict(batch=3, seqlen=130, heads_q=2, heads_kv=2, head_dim=128, causal=False),
    dict(batch=1, seqlen=1, heads_q=1, heads_kv=1, head_dim=128, causal=True),
])
@pytest.mark.parametrize("tau", [8.0, 0.0])
def test_fwd_edge_shapes(L, case, tau):
    """Ragged tails, GQA, head_dim 64, single token, and threshold 0 (the O
    correction path runs on every tile where the max grows)."""
    w = workloads.custom(seed=11, **case)
    x = workloads.make_inputs(w, with_grad_out=False)
    x["q"] = (x["q"].float() * 2).to(torch.bfloat16)   # move the max around
    o, lse = _run(L, x, w, tau)
    ref = A.mx_attention_fwd(x["q"], x["k"], x["v"], causal=w.causal,
                             softmax_scale=w.softmax_scale,
                             rescale_threshold=tau, kv_tile=A.FWD_KEY_TILE)
    assert relfro(o, ref["o"]) <= TOL_O
    assert np.abs(lse - ref["lse"]).max() <= TOL_LSE


def test_fwd_varlen_causal_ragged(L):
    lengths = torch.tensor([1, 127, 128, 129, 300, 64])
    cu = torch.zeros(7, dtype=torch.int32); cu[1:] = torch.cumsum(lengths, 0)
    T = int(cu[-1])
    g = torch.Generator().manual_seed(5)
    q = torch.randn(T, 4, 128, generator=g).to(torch.bfloat16)
    k = torch.randn(T, 2, 128, generator=g).to(torch.bfloat16)
    v = torch.randn(T, 2, 128, generator=g).to(torch.bfloat16)
    o, lse = L.mx_attention_forward(q.cuda(), k.cuda(), v.cuda(), causal=True,
                                    cu_seqlens=cu)
    torch.cuda.synchronize()
    ref = A.mx_attention_fwd(q, k, v, causal=True, softmax_scale=1 / math.sqrt(128),
                             cu_seqlens=cu.numpy(), kv_tile=A.FWD_KEY_TILE)
    assert relfro(o.float().cpu().numpy(), ref["o"]) <= TOL_O
    assert np.abs(lse.cpu().numpy() - ref["lse"]).max() <= TOL_LSE


def test_fwd_deterministic(L):
    w = workloads.get_config("outlier")
    x = workloads.make_inputs(w, with_grad_out=False)
    o1, l1 = _run(L, x, w)
    o2, l2 = _run(L, x, w)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
