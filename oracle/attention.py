"""Attention oracles in fp64: exact softmax attention, and MXFP8 block-scaled
attention at the quantization points the pages define.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``): imported by ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline legs, never by the
product path.

Sources
-------
[P1] "Low Precision Flash Attention 4: End-to-End Block-Scaled Attention for
     Blackwell" (aivexanews): paragraph 2 (block-scaled tcgen05 MMAs, online
     square-block quantization of dS, jagged module with 128-aligned scale
     rows), paragraph 3 (forward: softmax in FP32, P converted to MXFP8 with
     scales that reuse the softmax max; backward: Q, K, dO quantized in square
     [32, 32] blocks; FP16 dQ with a static scale).
[P2] "Low-Precision FlashAttention-4: End-to-End Block-Scaled Attention for
     NVIDIA Blackwell" (n1n.ai), "Key Algorithmic Innovations" 1-2: both GEMMs
     (QK^T and PV) are block-scaled MXFP8; the running max m_i and running sum
     l_i are kept in FP32 with 1/sqrt(d_k) folded in; "PyTorch Integration"
     example: BSHD tensors, softmax_scale, causal.
[P3] "FlashAttention-4 Adds Low-Precision Blackwell Support" (setupai),
     "Technical Deep Dive": selective rescaling of the output accumulator.

Readings (where the pages leave a step open):
* Forward blocks: Q and K are 1x32-blocked along head_dim; V is blocked in 32
  consecutive keys per head_dim column, because the PV product contracts over
  keys and a block-scaled MMA needs one scale per 32 elements of the
  contraction.  P is 1x32-blocked along keys, blocks aligned to the key tile.
* "Reusing the max already computed for softmax": P is quantized as the
  online softmax produces it, i.e. relative to the running reference max of
  the key tile being processed.  The oracle therefore runs the blockwise
  online algorithm over key tiles of ``kv_tile`` keys, with FA4's selective
  rescaling: the reference max m moves to the tile's row max only when that
  exceeds m by more than ``rescale_threshold`` (log2 units; 0 gives the
  classic online softmax).  l accumulates the unquantized FP32-path P.
* LSE is natural-log: ln(sum_j exp(c * s_ij)).
* Backward: Q, K, dO in 32x32 blocks over (token, head_dim); V in 1x32 blocks
  along head_dim (contraction of dP = dO V^T); P and dS in 32x32 blocks over
  (query, key).  D_i = sum_d dO_id * O_id from the bf16 O and dO.  c (the
  softmax scale) multiplies the dK and dQ accumulators after the quantized
  products.  dQ is accumulated in FP16: each 128-key tile's partial, times
  ``dq_static_scale``, is rounded to fp16 and added to an fp16 running sum in
  ascending tile order, and the sum is divided by the scale at the end.
* Causal masking keeps key j <= query i (Sq == Sk in every causal case, so
  top-left and bottom-right alignment coincide).
* GQA: query head h reads kv head h // (Hq / Hkv); dK, dV sum over the group.
* Varlen: every sequence is its own attention problem; blocks along tokens
  start at the sequence start and the last one may be short.
"""
from __future__ import annotations

import math

import numpy as np

from . import mx

LOG2E = 1.0 / math.log(2.0)
LN2 = math.log(2.0)

#: Keys per tile of the forward's online softmax.  With selective rescaling
#: the reference max, and with it the E4M3 rounding of P, moves at most once
#: per tile, so the quantization points of P depend on this length.  Reading
#: of "Low Precision Flash Attention 4 ...", paragraph 3 (P quantized with the
#: max the softmax already holds): one tile is 256 keys.
FWD_KEY_TILE = 256

#: Keys per FP16 dQ partial in the backward (each partial, times the static
#: scale, is rounded to FP16 and added to the FP16 dQ): 128 keys.
BWD_KEY_TILE = 128


# ----------------------------------------------------------------------------
# helpers: layouts
# ----------------------------------------------------------------------------
def to_f64(t) -> np.ndarray:
    """bf16/fp32 torch tensor or array -> fp64 numpy (exact)."""
    try:
        import torch
        if isinstance(t, torch.Tensor):
            return t.detach().to(torch.float64).cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(t, dtype=np.float64)


def _lazy(t):
    """Keep torch tensors as they are (sliced before conversion to fp64);
    other inputs become fp64 arrays."""
    try:
        import torch
        if isinstance(t, torch.Tensor):
            return t.detach().cpu()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(t, dtype=np.float64)


def as_packed(x, cu_seqlens):
    """[B, S, H, D] -> ([B*S, H, D], cu_seqlens); [T, H, D] passes through."""
    if x.ndim == 4:
        b, s = x.shape[:2]
        cu = np.arange(b + 1, dtype=np.int64) * s
        return x.reshape(b * s, *x.shape[2:]), cu
    assert cu_seqlens is not None
    return x, np.asarray(cu_seqlens, dtype=np.int64)


def _causal_mask(nq, nk, q0=0, k0=0):
    """True where key index (k0 + j) > query index (q0 + i)."""
    qi = q0 + np.arange(nq)[:, None]
    kj = k0 + np.arange(nk)[None, :]
    return kj > qi


# ----------------------------------------------------------------------------
# exact (unquantized) attention
# ----------------------------------------------------------------------------
def exact_fwd_head(q, k, v, causal, scale):
    """softmax(scale * q k^T) v for one head, fp64.  Returns (O, LSE)."""
    s = scale * (q @ k.T)
    if causal:
        s = np.where(_causal_mask(*s.shape), -np.inf, s)
    m = s.max(axis=1, keepdims=True)
    p = np.exp(s - m)
    l = p.sum(axis=1, keepdims=True)
    return (p / l) @ v, (m + np.log(l))[:, 0]


def exact_bwd_head(q, k, v, do, causal, scale):
    """Gradients of <dO, O> for one head from the softmax definition."""
    s = scale * (q @ k.T)
    if causal:
        s = np.where(_causal_mask(*s.shape), -np.inf, s)
    m = s.max(axis=1, keepdims=True)
    p = np.exp(s - m)
    p /= p.sum(axis=1, keepdims=True)
    o = p @ v
    dv = p.T @ do
    dp = do @ v.T
    delta = (do * o).sum(axis=1, keepdims=True)
    ds = p * (dp - delta)
    return scale * ds @ k, scale * ds.T @ q, dv


def exact_fwd_head_chunked(q, k, v, causal, scale, chunk=2048):
    """``exact_fwd_head`` computed over blocks of ``chunk`` query rows, so
    that long sequences need O(chunk * L) memory.  Query row i of the block
    starting at r0 is row r0 + i of the head; the causal mask keeps keys
    j <= r0 + i."""
    L = q.shape[0]
    o = np.empty((L, v.shape[1]))
    lse = np.empty(L)
    for r0 in range(0, L, chunk):
        r1 = min(r0 + chunk, L)
        kend = r1 if causal else k.shape[0]
        s = scale * (q[r0:r1] @ k[:kend].T)
        if causal:
            s = np.where(_causal_mask(r1 - r0, kend, q0=r0), -np.inf, s)
        m = s.max(axis=1, keepdims=True)
        p = np.exp(s - m)
        l = p.sum(axis=1, keepdims=True)
        o[r0:r1] = (p / l) @ v[:kend]
        lse[r0:r1] = (m + np.log(l))[:, 0]
    return o, lse


def exact_attention(q, k, v, *, causal, softmax_scale, cu_seqlens=None,
                    do=None):
    """Exact attention over packed or BSHD inputs (fp64).  Returns a dict with
    O (same layout as q), LSE [Hq, T], and dQ/dK/dV when ``do`` is given."""
    q = to_f64(q); k = to_f64(k); v = to_f64(v)
    shape_q, shape_k = q.shape, k.shape
    qp, cu = as_packed(q, cu_seqlens)
    kp, _ = as_packed(k, cu_seqlens)
    vp, _ = as_packed(v, cu_seqlens)
    hq, hkv = qp.shape[1], kp.shape[1]
    grp = hq // hkv
    o = np.zeros_like(qp)
    lse = np.zeros((hq, qp.shape[0]))
    res = {}
    if do is not None:
        dop, _ = as_packed(to_f64(do), cu_seqlens)
        dq = np.zeros_like(qp); dk = np.zeros_like(kp); dv = np.zeros_like(vp)
    for s in range(len(cu) - 1):
        a, b = cu[s], cu[s + 1]
        for h in range(hq):
            kh = h // grp
            oh, lh = exact_fwd_head(qp[a:b, h], kp[a:b, kh], vp[a:b, kh],
                                    causal, softmax_scale)
            o[a:b, h] = oh
            lse[h, a:b] = lh
            if do is not None:
                g = exact_bwd_head(qp[a:b, h], kp[a:b, kh], vp[a:b, kh],
                                   dop[a:b, h], causal, softmax_scale)
                dq[a:b, h] += g[0]; dk[a:b, kh] += g[1]; dv[a:b, kh] += g[2]
    res["o"] = o.reshape(shape_q)
    res["lse"] = lse
    if do is not None:
        res["dq"] = dq.reshape(shape_q)
        res["dk"] = dk.reshape(shape_k)
        res["dv"] = dv.reshape(shape_k)
    return res


# ----------------------------------------------------------------------------
# MXFP8 forward (quantization-matched)
# ----------------------------------------------------------------------------
def quantize_fwd_operands(qp, kp, vp, cu, quantize=True):
    """Dequantized fp64 copies of the forward operands: Q, K 1x32 along
    head_dim; V in 32-key blocks per head_dim column, per sequence."""
    if not quantize:
        return qp, kp, vp
    qd = mx.fake_quant_1x32(qp)
    kd = mx.fake_quant_1x32(kp)
    vd = np.empty_like(vp)
    for s in range(len(cu) - 1):
        a, b = cu[s], cu[s + 1]
        vd[a:b] = mx.fake_quant_rows(vp[a:b])
    return qd, kd, vd


def mx_fwd_head(q, k, v, *, causal, scale, kv_tile=FWD_KEY_TILE, rescale_threshold=8.0,
                quantize=True, rows=None):
    """Blockwise online softmax attention for one head of one sequence.

    q, k, v are the (already dequantized) operands [L, D].  ``rows`` selects
    query rows (default all); rows are independent in the algorithm.
    Returns (O [nrows, D], LSE [nrows])."""
    L = k.shape[0]
    if rows is None:
        rows = np.arange(q.shape[0])
    qr = q[rows]
    n = qr.shape[0]
    c2 = scale * LOG2E                      # logits in log2 units
    m_ref = np.full(n, -np.inf)
    l = np.zeros(n)
    acc = np.zeros((n, v.shape[1]))
    for t0 in range(0, L, kv_tile):
        t1 = min(t0 + kv_tile, L)
        x = c2 * (qr @ k[t0:t1].T)          # [n, tile]
        if causal:
            masked = (t0 + np.arange(t1 - t0))[None, :] > rows[:, None]
            x = np.where(masked, -np.inf, x)
        else:
            masked = np.zeros(x.shape, dtype=bool)
        mt = x.max(axis=1)
        move = (mt > m_ref + rescale_threshold) | np.isneginf(m_ref)
        m_new = np.where(move, mt, m_ref)
        finite = np.isfinite(m_new)
        alpha = np.where(np.isfinite(m_ref) & finite,
                         np.exp2(np.where(finite, m_ref - m_new, 0.0)), 0.0)
        p = np.where(masked | ~finite[:, None], 0.0,
                     np.exp2(x - np.where(finite, m_new, 0.0)[:, None]))
        if quantize:
            w = t1 - t0
            wpad = -(-w // 32) * 32
            pp = np.concatenate([p, np.zeros((n, wpad - w))], 1) if wpad > w else p
            p_hat = mx.fake_quant_1x32(pp)[:, :w]
        else:
            p_hat = p
        acc = alpha[:, None] * acc + p_hat @ v[t0:t1]
        l = alpha * l + p.sum(axis=1)
        m_ref = m_new
    o = acc / l[:, None]
    lse = m_ref * LN2 + np.log(l)
    return o, lse


def mx_attention_fwd(q, k, v, *, causal, softmax_scale, cu_seqlens=None,
                     kv_tile=FWD_KEY_TILE, rescale_threshold=8.0, quantize=True,
                     heads=None, seqs=None, rows=None):
    """MXFP8 block-scaled attention forward over packed [T, H, D] (with
    ``cu_seqlens``) or BSHD inputs.

    ``heads`` / ``seqs`` / ``rows`` restrict the work to a sample (query heads,
    sequence indices, query rows within each sequence); entries outside the
    sample are NaN.  Returns {"o": like q, "lse": [Hq, T]}."""
    shape_q = tuple(q.shape)
    hq, hkv = q.shape[-2], k.shape[-2]
    grp = hq // hkv
    qp, cu = as_packed(_lazy(q), cu_seqlens)
    kp, _ = as_packed(_lazy(k), cu_seqlens)
    vp, _ = as_packed(_lazy(v), cu_seqlens)
    T = qp.shape[0]
    o = np.full((T, hq, qp.shape[2]), np.nan)
    lse = np.full((hq, T), np.nan)
    heads = range(hq) if heads is None else heads
    seqs = range(len(cu) - 1) if seqs is None else seqs
    for s in seqs:
        a, b = cu[s], cu[s + 1]
        r = np.arange(b - a) if rows is None else np.asarray(
            [i for i in rows if i < b - a], dtype=np.int64)
        for h in heads:
            kh = h // grp
            # operands of this (sequence, head) only; quantization acts per
            # row (Q, K) or per 32-token block of one sequence (V)
            qd, kd, vd = quantize_fwd_operands(
                to_f64(qp[a:b, h:h + 1]), to_f64(kp[a:b, kh:kh + 1]),
                to_f64(vp[a:b, kh:kh + 1]), np.array([0, b - a]), quantize)
            oh, lh = mx_fwd_head(qd[:, 0], kd[:, 0], vd[:, 0],
                                 causal=causal, scale=softmax_scale,
                                 kv_tile=kv_tile,
                                 rescale_threshold=rescale_threshold,
                                 quantize=quantize, rows=r)
            o[a + r, h] = oh
            lse[h, a + r] = lh
    return {"o": o.reshape(shape_q), "lse": lse}


# ----------------------------------------------------------------------------
# MXFP8 backward (quantization-matched)
# ----------------------------------------------------------------------------
def _fp16(x):
    return np.asarray(x, dtype=np.float64).astype(np.float16)


def _square_per_head(x):
    """32x32 blocks over (token, head_dim) of x [L, H, D], for every head."""
    xt = np.moveaxis(x, 2, 1)                   # [L, D, H]
    return np.moveaxis(mx.fake_quant_32x32(xt), 1, 2)


def quantize_bwd_operands(qp, kp, vp, dop, cu, quantize=True):
    """Dequantized backward operands: Q, K, dO in 32x32 blocks over
    (token, head_dim) per sequence and head; V 1x32 along head_dim."""
    if not quantize:
        return qp, kp, vp, dop
    out = []
    for x in (qp, kp, dop):
        y = np.empty_like(x)
        for s in range(len(cu) - 1):
            a, b = cu[s], cu[s + 1]
            y[a:b] = _square_per_head(x[a:b])
        out.append(y)
    qd, kd, dod = out
    vd = mx.fake_quant_1x32(vp)
    return qd, kd, vd, dod


def _square_on_grid(x, fq):
    """32x32 block quantization of a sub-grid x whose rows and columns are
    whole 32-aligned blocks of the full (query, key) grid, in order, the last
    block possibly short.  Columns are zero-padded to a multiple of 32."""
    w = x.shape[1]
    wpad = -(-w // 32) * 32
    if wpad > w:
        x = np.concatenate([x, np.zeros((x.shape[0], wpad - w))], 1)
    return fq(x)[:, :w]


def _check_whole_blocks(idx, L):
    idx = np.asarray(idx, dtype=np.int64)
    if idx.size == 0:
        return idx
    assert np.all(np.diff(idx) > 0)
    for b in np.unique(idx // 32):
        want = np.arange(32 * b, min(32 * b + 32, L))
        got = idx[(idx // 32) == b]
        assert got.size == want.size and np.all(got == want), \
            "row samples must be whole 32-row blocks"
    return idx


def mx_bwd_head(q, k, v, dod, do_raw, o, lse, *, causal, scale, quantize=True,
                kv_tile=BWD_KEY_TILE, dq_static_scale=1.0, q_rows=None,
                k_rows=None):
    """Backward for one head of one sequence.

    q, k, v, dod: dequantized operands [L, D]; do_raw and o: the bf16-valued
    dO and forward output (for D_i); lse [L]: forward log-sum-exp (natural).
    ``q_rows`` selects the dQ rows, ``k_rows`` the dK/dV rows (whole 32-row
    blocks).  Rows of o/lse that cannot see a selected key are not read.
    Returns (dQ [q_rows, D] (FP16-accumulated), dK [k_rows, D], dV)."""
    L = q.shape[0]
    q_rows = _check_whole_blocks(np.arange(L) if q_rows is None else q_rows, L)
    k_rows = _check_whole_blocks(np.arange(L) if k_rows is None else k_rows, L)

    def fq(x):
        return mx.fake_quant_32x32(x) if quantize else x

    def p_ds(qi, kj):
        """P = exp(c*S - LSE) and dS = P * (dP - D) on the (qi, kj) grid."""
        s = scale * (q[qi] @ k[kj].T)
        dp = dod[qi] @ v[kj].T
        delta = (do_raw[qi] * o[qi]).sum(axis=1)            # D_i
        mask = (kj[None, :] > qi[:, None]) if causal else np.zeros(s.shape, bool)
        p = np.where(mask, 0.0, np.exp(np.where(mask, 0.0, s - lse[qi][:, None])))
        ds = p * (dp - delta[:, None])
        return p, ds

    D = q.shape[1]
    dk = np.zeros((len(k_rows), D)); dv = np.zeros((len(k_rows), D))
    if len(k_rows):
        # queries that can attend to any selected key (whole 32-row blocks)
        q0 = (int(k_rows.min()) // 32) * 32 if causal else 0
        qi = np.arange(q0, L)
        p, ds = p_ds(qi, k_rows)
        p_hat = _square_on_grid(p, fq)
        ds_hat = _square_on_grid(ds, fq)
        dv = p_hat.T @ dod[qi]
        dk = scale * (ds_hat.T @ q[qi])
    acc = np.zeros((len(q_rows), D), dtype=np.float16)
    if len(q_rows):
        kend = int(q_rows.max()) + 1 if causal else L
        kj = np.arange(0, kend)
        _, ds_q = p_ds(q_rows, kj)
        ds_q_hat = _square_on_grid(ds_q, fq)
        for t0 in range(0, kend, kv_tile):
            t1 = min(t0 + kv_tile, kend)
            part = scale * dq_static_scale * (ds_q_hat[:, t0:t1] @ k[t0:t1])
            acc = _fp16(acc.astype(np.float64) + _fp16(part).astype(np.float64))
    dq = acc.astype(np.float64) / dq_static_scale
    return dq, dk, dv


def mx_attention_bwd(q, k, v, o, do, lse, *, causal, softmax_scale,
                     cu_seqlens=None, kv_tile=BWD_KEY_TILE, dq_static_scale=1.0,
                     quantize=True, heads=None, seqs=None, q_rows=None,
                     k_rows=None):
    """MXFP8 block-scaled attention backward over packed or BSHD inputs.

    ``o`` is the forward output (bf16 values) and ``lse`` [Hq, T] the forward
    log-sum-exp that P is recomputed from.  ``heads`` restricts to kv heads
    (with all their query heads), ``seqs`` to sequences, ``q_rows``/``k_rows``
    to whole 32-row blocks within each sequence.  Entries outside the sample
    are NaN.  Returns {"dq", "dk", "dv"} shaped like q/k/v."""
    shape_q, shape_k = tuple(q.shape), tuple(k.shape)
    lse = to_f64(lse)
    qp, cu = as_packed(_lazy(q), cu_seqlens)
    kp, _ = as_packed(_lazy(k), cu_seqlens)
    vp, _ = as_packed(_lazy(v), cu_seqlens)
    op, _ = as_packed(_lazy(o), cu_seqlens)
    dop, _ = as_packed(_lazy(do), cu_seqlens)
    hq, hkv = qp.shape[1], kp.shape[1]
    grp = hq // hkv
    T, D = qp.shape[0], qp.shape[2]
    dq = np.full((T, hq, D), np.nan)
    dk = np.full((T, hkv, D), np.nan)
    dv = np.full((T, hkv, D), np.nan)
    kv_heads = range(hkv) if heads is None else heads
    seqs = range(len(cu) - 1) if seqs is None else seqs
    for s in seqs:
        a, b = cu[s], cu[s + 1]
        L = b - a
        qr = np.arange(L) if q_rows is None else np.asarray(
            [i for i in q_rows if i < L], dtype=np.int64)
        kr = np.arange(L) if k_rows is None else np.asarray(
            [i for i in k_rows if i < L], dtype=np.int64)
        one = np.array([0, L])
        for kh in kv_heads:
            dk_acc = np.zeros((len(kr), D))
            dv_acc = np.zeros((len(kr), D))
            for h in range(kh * grp, (kh + 1) * grp):
                qd, kd, vd, dod = quantize_bwd_operands(
                    to_f64(qp[a:b, h:h + 1]), to_f64(kp[a:b, kh:kh + 1]),
                    to_f64(vp[a:b, kh:kh + 1]), to_f64(dop[a:b, h:h + 1]),
                    one, quantize)
                g = mx_bwd_head(qd[:, 0], kd[:, 0], vd[:, 0], dod[:, 0],
                                to_f64(dop[a:b, h]), to_f64(op[a:b, h]),
                                lse[h, a:b], causal=causal,
                                scale=softmax_scale, quantize=quantize,
                                kv_tile=kv_tile,
                                dq_static_scale=dq_static_scale,
                                q_rows=qr, k_rows=kr)
                dq[a + qr, h] = g[0]
                dk_acc += g[1]
                dv_acc += g[2]
            dk[a + kr, kh] = dk_acc
            dv[a + kr, kh] = dv_acc
    return {"dq": dq.reshape(shape_q), "dk": dk.reshape(shape_k),
            "dv": dv.reshape(shape_k)}
