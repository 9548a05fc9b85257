"""Backward parity on the GPU against the quantization-matched oracle
(dQ, dK, dV relative Frobenius <= 5e-2).  Two forms: the GPU forward's O and
LSE feed the GPU backward while the oracle runs its own forward (end-to-end
training path), and both backwards get the oracle's O / LSE (isolates the
backward kernel)."""
import numpy as np
import pytest
import torch

import workloads
from oracle import attention as A

pytestmark = pytest.mark.gpu

TOL = 5e-2


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


def _gpu_fwd_bwd(L, x, w, dq_scale=1.0):
    cu = x["cu_seqlens"] if w.varlen else None
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = L.mx_attention_forward(q, k, v, causal=w.causal,
                                    softmax_scale=w.softmax_scale, cu_seqlens=cu)
    dq, dk, dv = L.mx_attention_backward(q, k, v, o, do, lse, causal=w.causal,
                                         softmax_scale=w.softmax_scale,
                                         cu_seqlens=cu, dq_static_scale=dq_scale)
    torch.cuda.synchronize()
    return [t.float().cpu().numpy() for t in (dq, dk, dv)]


def _oracle(x, w, heads=None, seqs=None, q_rows=None, k_rows=None,
            fwd_rows=None, dq_scale=1.0):
    """Oracle forward (its own O, LSE) then backward on a sample: ``heads``
    are kv heads (all their query heads are computed)."""
    cu = x["cu_seqlens"].numpy() if w.varlen else None
    grp = w.heads_q // w.heads_kv
    qheads = None if heads is None else \
        [h for kh in heads for h in range(kh * grp, (kh + 1) * grp)]
    fw = A.mx_attention_fwd(x["q"], x["k"], x["v"], causal=w.causal,
                            softmax_scale=w.softmax_scale, cu_seqlens=cu,
                            seqs=seqs, rows=fwd_rows, heads=qheads, kv_tile=A.FWD_KEY_TILE)
    o16 = torch.from_numpy(np.nan_to_num(fw["o"])).to(torch.bfloat16)
    bw = A.mx_attention_bwd(x["q"], x["k"], x["v"], o16, x["do"],
                            np.nan_to_num(fw["lse"]), causal=w.causal,
                            softmax_scale=w.softmax_scale, cu_seqlens=cu,
                            heads=heads, seqs=seqs, q_rows=q_rows, k_rows=k_rows,
                            dq_static_scale=dq_scale)
    return bw, o16, fw["lse"]


def _check(got, ref, sel_q, sel_k, tag, names=("dq", "dk", "dv")):
    for name, g, r, sel in (("dq", got[0], ref["dq"], sel_q),
                            ("dk", got[1], ref["dk"], sel_k),
                            ("dv", got[2], ref["dv"], sel_k)):
        if name not in names:
            continue
        gt, rt = _tok(g), _tok(r)
        e = relfro(gt[sel], rt[sel])
        assert e <= TOL, f"{tag} {name}: {e:.3e}"


def test_bwd_isolated_with_oracle_forward(L):
    """Both backwards see the oracle's O and LSE."""
    w = workloads.custom(seed=4, batch=2, seqlen=1024, heads_q=4, heads_kv=4,
                         head_dim=128, causal=True)
    x = workloads.make_inputs(w)
    ref, o16, lse = _oracle(x, w, heads=[3])
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    lse_in = torch.from_numpy(np.nan_to_num(lse)).float().cuda()
    dq, dk, dv = L.mx_attention_backward(q, k, v, o16.cuda(), do, lse_in,
                                         causal=True,
                                         softmax_scale=w.softmax_scale)
    torch.cuda.synchronize()
    got = [t.float().cpu().numpy() for t in (dq, dk, dv)]
    S = w.seqlen
    for b in range(w.batch):
        rows = (slice(b * S, (b + 1) * S), 3)
        _check(got, ref, rows, rows, f"isolated b{b}")
        for name, g, r in (("dk", got[1], ref["dk"]), ("dv", got[2], ref["dv"])):
            assert relfro(_tok(g)[rows], _tok(r)[rows]) < 1e-2, name


def test_bwd_tiny_full(L):
    """Tiny workload (head_dim 64, non-causal), every output compared."""
    w = workloads.get_config("tiny")
    x = workloads.make_inputs(w)
    got = _gpu_fwd_bwd(L, x, w)
    ref, _, _ = _oracle(x, w)
    allr = (slice(None),)
    _check(got, ref, allr, allr, "tiny")


@pytest.mark.parametrize("case", [
    dict(batch=2, seqlen=200, heads_q=4, heads_kv=1, head_dim=128, causal=True),
    dict(batch=2, seqlen=333, heads_q=4, heads_kv=2, head_dim=64, causal=True),
    dict(batch=1, seqlen=320, heads_q=2, heads_kv=2, head_dim=128, causal=False),
    dict(batch=1, seqlen=1, heads_q=1, heads_kv=1, head_dim=128, causal=True),
    dict(batch=3, seqlen=96, heads_q=2, heads_kv=2, head_dim=128, causal=True),
])
def test_bwd_edge_shapes(L, case):
    """Ragged tails, GQA 4:1, non-causal, a single token."""
    w = workloads.custom(seed=21, **case)
    x = workloads.make_inputs(w)
    got = _gpu_fwd_bwd(L, x, w)
    ref, _, _ = _oracle(x, w)
    allr = (slice(None),)
    _check(got, ref, allr, allr, str(case))


def test_bwd_outlier_sampled_heads(L):
    """Outlier workload.  Its logits reach ~70 standard deviations, so the
    backward's logits (Q, K in 32x32 blocks) differ from the forward's (1x32
    blocks) by tens in log space and P = exp(c S - LSE) grows far above 1 in
    the oracle as in the kernel; FP16 dQ then overflows on some rows.  dK and
    dV stay finite and are compared in full; dQ on the rows where the
    oracle's FP16 dQ is finite, and the kernel must be non-finite wherever
    the oracle overflowed."""
    w = workloads.get_config("outlier")
    x = workloads.make_inputs(w)
    got = _gpu_fwd_bwd(L, x, w)
    heads = [0, 15]
    with np.errstate(over="ignore", invalid="ignore"):
        ref, _, _ = _oracle(x, w, heads=heads)
    S = w.seqlen
    dq_g, dq_r = _tok(got[0]), _tok(ref["dq"])
    for b in range(w.batch):
        for h in heads:
            rows = (slice(b * S, (b + 1) * S), h)
            _check(got, ref, None, rows, f"b{b}h{h}", names=("dk", "dv"))
            fin = np.all(np.isfinite(dq_r[rows]), axis=1)
            assert fin.mean() > 0.5
            e = relfro(dq_g[rows][fin], dq_r[rows][fin])
            assert e <= TOL, f"b{b}h{h} dq(finite rows): {e:.3e}"
            assert not np.any(np.all(np.isfinite(dq_g[rows][~fin]), axis=1))


@pytest.mark.parametrize("name", ["llm", "gqa_long"])
def test_bwd_full_size_sampled(L, name):
    """Full-size launch; oracle on the last 128 keys / queries of the first
    and last sequence for the first and last kv head."""
    w = workloads.get_config(name)
    x = workloads.make_inputs(w)
    got = _gpu_fwd_bwd(L, x, w)
    S = w.seqlen
    rows = np.arange(S - 128, S)
    heads = [0, w.heads_kv - 1]
    seqs = [0, w.batch - 1]
    ref, _, _ = _oracle(x, w, heads=heads, seqs=seqs, q_rows=rows,
                        k_rows=rows, fwd_rows=rows)
    grp = w.heads_q // w.heads_kv
    for b in seqs:
        for kh in heads:
            kr = (b * S + rows, kh)
            qr = (b * S + rows, kh * grp)
            _check(got, ref, qr, kr, f"{name} b{b} kv{kh}")


def test_bwd_full_size_first_key_tile_end_to_end(L):
    """llm, last sequence and head: the first 128 keys are seen by all 8192
    queries (the longest query loop of the causal backward, 128 steps); their
    dK, dV and the first 128 rows of dQ against the oracle running its own
    forward over every query row."""
    w = workloads.get_config("llm")
    x = workloads.make_inputs(w)
    got = _gpu_fwd_bwd(L, x, w)
    S, b, kh = w.seqlen, w.batch - 1, w.heads_kv - 1
    rows = np.arange(0, 128)
    ref, _, _ = _oracle(x, w, heads=[kh], seqs=[b], q_rows=rows, k_rows=rows)
    sel = (b * S + rows, kh)
    _check(got, ref, sel, sel, "llm first key tile")


@pytest.mark.parametrize("name,pairs", [("llm", [(0, 0), (7, 31)]),
                                        ("gqa_long", [(0, 7)])])
def test_bwd_full_size_isolated(L, name, pairs):
    """Isolated form at full size: both backwards get the same O and LSE,
    the oracle's exact fp64 attention of the sampled (sequence, kv head)
    pairs (all query heads of the group; other heads keep the GPU forward's
    O and LSE and are not compared).  Compared: the first and the last 128
    keys (dK, dV: the longest and the shortest causal query loops, 512 steps
    per query head for the first key tile of gqa_long) and the first and last
    128 query rows of dQ."""
    w = workloads.get_config(name)
    x = workloads.make_inputs(w)
    S, D = w.seqlen, w.head_dim
    grp = w.heads_q // w.heads_kv
    T = w.batch * S
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = L.mx_attention_forward(q, k, v, causal=True,
                                    softmax_scale=w.softmax_scale)
    # the oracle's inputs hold only oracle values (zeros elsewhere)
    o_or = torch.zeros(T, w.heads_q, D, dtype=torch.bfloat16)
    lse_or = np.zeros((w.heads_q, T))
    qt, kt, vt = (_tok(x[n]) for n in ("q", "k", "v"))
    for b, kh in pairs:
        for h in range(kh * grp, (kh + 1) * grp):
            oh, lh = A.exact_fwd_head_chunked(
                qt[b * S:(b + 1) * S, h].double().numpy(),
                kt[b * S:(b + 1) * S, kh].double().numpy(),
                vt[b * S:(b + 1) * S, kh].double().numpy(), True, w.softmax_scale)
            o_or[b * S:(b + 1) * S, h] = torch.from_numpy(oh).to(torch.bfloat16)
            lse_or[h, b * S:(b + 1) * S] = lh
            o.view(T, w.heads_q, D)[b * S:(b + 1) * S, h] = \
                o_or[b * S:(b + 1) * S, h].cuda()
            lse[h, b * S:(b + 1) * S] = torch.from_numpy(lh).float().cuda()
    dq, dk, dv = L.mx_attention_backward(q, k, v, o, do, lse, causal=True,
                                         softmax_scale=w.softmax_scale)
    torch.cuda.synchronize()
    got = [t.float().cpu().numpy() for t in (dq, dk, dv)]
    rows = np.concatenate([np.arange(0, 128), np.arange(S - 128, S)])
    shape = x["q"].shape
    for b, kh in pairs:
        ref = A.mx_attention_bwd(x["q"], x["k"], x["v"], o_or.reshape(shape),
                                 x["do"], lse_or, causal=True,
                                 softmax_scale=w.softmax_scale, heads=[kh],
                                 seqs=[b], q_rows=rows, k_rows=rows)
        for part in (rows[:128], rows[128:]):
            kr = (b * S + part, kh)
            for h in range(kh * grp, (kh + 1) * grp):
                _check(got, ref, (b * S + part, h), kr,
                       f"{name} b{b} kv{kh} h{h} rows {part[0]}..")


def test_bwd_varlen_sampled_sequences(L):
    w = workloads.get_config("varlen")
    x = workloads.make_inputs(w)
    got = _gpu_fwd_bwd(L, x, w)
    lens = x["lengths"].numpy()
    cu = x["cu_seqlens"].numpy()
    seqs = sorted({int(lens.argmin()), int(lens.argmax()), 9})
    heads = [0, 15]
    ref, _, _ = _oracle(x, w, heads=heads, seqs=seqs)
    for s in seqs:
        for h in heads:
            sel = (slice(cu[s], cu[s + 1]), h)
            _check(got, ref, sel, sel, f"seq{s} h{h}")


def test_bwd_dq_static_scale(L):
    """dq_static_scale = 8 against the oracle at the same scale (FP16
    partials times 8, divided out at the end); dK and dV do not depend on it."""
    w = workloads.custom(seed=3, batch=1, seqlen=256, heads_q=2, heads_kv=2,
                         head_dim=128, causal=True)
    x = workloads.make_inputs(w)
    g1 = _gpu_fwd_bwd(L, x, w, 1.0)
    g8 = _gpu_fwd_bwd(L, x, w, 8.0)
    ref8, _, _ = _oracle(x, w, dq_scale=8.0)
    allr = (slice(None),)
    _check(g8, ref8, allr, allr, "dq_static_scale=8")
    assert np.array_equal(g8[1], g1[1]) and np.array_equal(g8[2], g1[2])
