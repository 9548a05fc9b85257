"""The bf16 variants of the attention kernels against exact fp64 attention.

The bf16 forward computes S = c q k^T exactly in fp32 from bf16 inputs (each
product of two bf16 values is exact in fp32), keeps the softmax in fp32, and
rounds only P (to bf16, for the PV product) and O (to bf16): each of these
roundings is within 2^-9 relative, so O lies within about 2^-8 of the exact
result element by element and its relative Frobenius error stays near
2^-9.  Tolerances: O relative Frobenius <= 5e-3, LSE absolute <= 1e-3.
"""
import numpy as np
import pytest
import torch

import workloads
from oracle import attention as A

pytestmark = pytest.mark.gpu

TOL_O, TOL_LSE = 5e-3, 1e-3


@pytest.fixture(scope="module")
def L():
    from mxfp8_block_scaled_quantizer_gb300 import build
    build()
    from mxfp8_block_scaled_quantizer_gb300 import lpfa
    return lpfa


def relfro(a, b):
    a = np.asarray(a, np.float64); b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def _tok(a):
    return a.reshape(-1, *a.shape[2:]) if a.ndim == 4 else a


def _fwd(L, x, w):
    cu = x["cu_seqlens"] if w.varlen else None
    o, lse = L.bf16_attention_forward(x["q"].cuda(), x["k"].cuda(), x["v"].cuda(),
                                      causal=w.causal, softmax_scale=w.softmax_scale,
                                      cu_seqlens=cu)
    torch.cuda.synchronize()
    return _tok(o.float().cpu().numpy()), lse.cpu().numpy()


def _exact_heads(x, w, pairs):
    """Exact attention of (sequence, query head) pairs: {pair: (O, LSE)}."""
    qt, kt, vt = (_tok(x[n]) for n in ("q", "k", "v"))
    cu = x["cu_seqlens"].numpy() if w.varlen else \
        np.arange(w.batch + 1) * w.seqlen
    grp = w.heads_q // w.heads_kv
    out = {}
    for s, h in pairs:
        a, b = cu[s], cu[s + 1]
        out[(s, h)] = A.exact_fwd_head_chunked(
            qt[a:b, h].double().numpy(), kt[a:b, h // grp].double().numpy(),
            vt[a:b, h // grp].double().numpy(), w.causal, w.softmax_scale)
    return out, cu


def _check(o, lse, ref, cu, tag):
    for (s, h), (ro, rl) in ref.items():
        a, b = cu[s], cu[s + 1]
        e = relfro(o[a:b, h], ro)
        assert e <= TOL_O, f"{tag} seq{s} h{h} O {e:.3e}"
        d = np.abs(lse[h, a:b] - rl).max()
        assert d <= TOL_LSE, f"{tag} seq{s} h{h} LSE {d:.3e}"


def test_bf16_fwd_tiny_full(L):
    w = workloads.get_config("tiny")
    x = workloads.make_inputs(w, with_grad_out=False)
    o, lse = _fwd(L, x, w)
    ref, cu = _exact_heads(x, w, [(0, h) for h in range(w.heads_q)])
    _check(o, lse, ref, cu, "tiny")


@pytest.mark.parametrize("case", [
    dict(batch=2, seqlen=200, heads_q=4, heads_kv=1, head_dim=128, causal=True),
    dict(batch=2, seqlen=333, heads_q=4, heads_kv=2, head_dim=64, causal=True),
    dict(batch=1, seqlen=320, heads_q=2, heads_kv=2, head_dim=128, causal=False),
    dict(batch=1, seqlen=1, heads_q=1, heads_kv=1, head_dim=128, causal=True),
    dict(batch=3, seqlen=700, heads_q=2, heads_kv=2, head_dim=64, causal=False),
])
def test_bf16_fwd_edge_shapes(L, case):
    """Ragged tails, GQA 4:1, head_dim 64, non-causal, a single token."""
    w = workloads.custom(seed=23, **case)
    x = workloads.make_inputs(w, with_grad_out=False)
    o, lse = _fwd(L, x, w)
    ref, cu = _exact_heads(x, w, [(s, h) for s in range(w.batch) for h in range(w.heads_q)])
    _check(o, lse, ref, cu, str(case))


@pytest.mark.parametrize("name", ["llm", "gqa_long"])
def test_bf16_fwd_full_size_sampled(L, name):
    """Full-size launch; exact attention of the first and last head of the
    first and last sequence."""
    w = workloads.get_config(name)
    x = workloads.make_inputs(w, with_grad_out=False)
    o, lse = _fwd(L, x, w)
    pairs = [(0, 0), (w.batch - 1, w.heads_q - 1)]
    ref, cu = _exact_heads(x, w, pairs)
    _check(o, lse, ref, cu, name)


def test_bf16_fwd_varlen_sampled(L):
    w = workloads.get_config("varlen")
    x = workloads.make_inputs(w, with_grad_out=False)
    o, lse = _fwd(L, x, w)
    lens = x["lengths"].numpy()
    seqs = sorted({int(lens.argmin()), int(lens.argmax()), 9})
    ref, cu = _exact_heads(x, w, [(s, h) for s in seqs for h in (0, 15)])
    _check(o, lse, ref, cu, "varlen")


# ------------------------------------------------------------------ backward
# The bf16 backward rounds P^T and dS^T to bf16 for their products (2^-9
# relative each), takes D_i from the bf16 O, accumulates dQ in FP16 (2^-11 per
# add) and writes dK, dV in bf16: against exact gradients of the same O and
# LSE, dQ, dK, dV relative Frobenius <= 1e-2.
TOL_G = 1e-2


def _grad_err(a, b):
    """Relative Frobenius error; a reference that is exactly zero (one key:
    dS = P (dP - D) vanishes) is compared in absolute terms instead."""
    nb = np.linalg.norm(b)
    if nb == 0.0:
        return float(np.abs(a).max()) / 1e-3
    return relfro(a, b)


def _bwd_case(L, x, w, pairs):
    """GPU bf16 backward with both sides given the exact O and LSE of the
    sampled (sequence, kv head) pairs (other heads: the bf16 forward's)."""
    qt, kt, vt, dot = (_tok(x[n]) for n in ("q", "k", "v", "do"))
    cu = x["cu_seqlens"] if w.varlen else None
    cu_np = cu.numpy() if w.varlen else np.arange(w.batch + 1) * w.seqlen
    grp = w.heads_q // w.heads_kv
    # BSHD for dense inputs, packed [T, H, D] with cu_seqlens for varlen
    dev = [x[n].cuda() for n in ("q", "k", "v", "do")]
    o4, lse = L.bf16_attention_forward(*dev[:3], causal=w.causal,
                                       softmax_scale=w.softmax_scale, cu_seqlens=cu)
    o = o4.view(qt.shape)
    want = {}
    for s, kh in pairs:
        a, b = cu_np[s], cu_np[s + 1]
        for h in range(kh * grp, (kh + 1) * grp):
            args = [t[a:b, hh].double().numpy() for t, hh in
                    ((qt, h), (kt, kh), (vt, kh), (dot, h))]
            oh, lh = A.exact_fwd_head(*args[:3], w.causal, w.softmax_scale)
            o16 = torch.from_numpy(oh).to(torch.bfloat16)
            o[a:b, h] = o16.cuda()
            lse[h, a:b] = torch.from_numpy(lh).float().cuda()
            # exact gradients of the same O (bf16 values) and LSE
            want[(s, h)] = A.exact_bwd_head(*args, w.causal, w.softmax_scale)
    dq, dk, dv = L.bf16_attention_backward(dev[0], dev[1], dev[2], o4, dev[3], lse,
                                           causal=w.causal, softmax_scale=w.softmax_scale,
                                           cu_seqlens=cu)
    torch.cuda.synchronize()
    got = [_tok(t.float().cpu().numpy()) for t in (dq, dk, dv)]
    for s, kh in pairs:
        a, b = cu_np[s], cu_np[s + 1]
        gk = np.zeros((b - a, w.head_dim)); gv = np.zeros((b - a, w.head_dim))
        for h in range(kh * grp, (kh + 1) * grp):
            e = _grad_err(got[0][a:b, h], want[(s, h)][0])
            assert e <= TOL_G, f"seq{s} h{h} dq {e:.3e}"
            gk += want[(s, h)][1]; gv += want[(s, h)][2]
        for name, g_, r_ in (("dk", got[1][a:b, kh], gk), ("dv", got[2][a:b, kh], gv)):
            e = _grad_err(g_, r_)
            assert e <= TOL_G, f"seq{s} kv{kh} {name} {e:.3e}"


@pytest.mark.parametrize("case", [
    dict(batch=2, seqlen=200, heads_q=4, heads_kv=1, causal=True),
    dict(batch=1, seqlen=320, heads_q=2, heads_kv=2, causal=False),
    dict(batch=3, seqlen=96, heads_q=2, heads_kv=2, causal=True),
    dict(batch=1, seqlen=1, heads_q=1, heads_kv=1, causal=True),
    dict(batch=1, seqlen=1000, heads_q=4, heads_kv=2, causal=True),
])
def test_bf16_bwd_edge_shapes(L, case):
    w = workloads.custom(seed=31, head_dim=128, **case)
    x = workloads.make_inputs(w)
    _bwd_case(L, x, w, [(s, kh) for s in range(w.batch) for kh in range(w.heads_kv)])


def test_bf16_bwd_full_size_sampled(L):
    """llm workload at full size, first and last (sequence, head)."""
    w = workloads.get_config("llm")
    x = workloads.make_inputs(w)
    _bwd_case(L, x, w, [(0, 0), (w.batch - 1, w.heads_kv - 1)])


def test_bf16_bwd_varlen_sampled(L):
    w = workloads.get_config("varlen")
    x = workloads.make_inputs(w)
    lens = x["lengths"].numpy()
    _bwd_case(L, x, w, [(int(lens.argmin()), 0), (int(lens.argmax()), 15)])


def test_bf16_bwd_rejects_head_dim_64(L):
    w = workloads.custom(seed=1, batch=1, seqlen=64, heads_q=1, heads_kv=1, head_dim=64,
                         causal=True)
    x = workloads.make_inputs(w)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    lse = torch.zeros((1, 64), dtype=torch.float32, device="cuda")
    with pytest.raises(L.LpfaError) as ei:
        L.bf16_attention_backward(q, k, v, do, do, lse, causal=True)
    assert ei.value.status == L.LPFA_ERR_UNSUPPORTED
