"""lpfa_bwd_noalloc: the backward for callers that cannot allocate device
memory (a runtime that owns every buffer, or code that must not call the
CUDA allocator because it can synchronise the device).  It keeps its scratch
in the library's static device array instead of a caller workspace.

The GPU test calls it through the C ABI twice in a row and compares each
result with lpfa_bwd's (same inputs, caller-allocated workspace): both run
the same kernel, whose dK and dV accumulate in a fixed order, so those must be
bit-identical; dQ is a sum of FP16 reduce-adds whose order varies from run to
run, so it must agree to within a few FP16 roundings.  The file is named so
that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads

# three 128-key partials per dQ element here, each add rounded to FP16
# (relative 2^-11): the two orders differ by a few units of that
DQ_TOL = 2e-3


@pytest.fixture(scope="module")
def L():
    from mxfp8_block_scaled_quantizer_gb300 import build
    build()
    from mxfp8_block_scaled_quantizer_gb300 import lpfa
    return lpfa


def _relfro(a, b):
    a = a.double(); b = b.double()
    return float((a - b).norm() / b.norm())


def test_noalloc_rejects_problems_beyond_the_scratch_size(L):
    """Too many (head, padded row) pairs for the static array: rejected on
    the host before any device work (runs without a GPU)."""
    rows = 1 << 24                      # 8 B/row of scratch -> 128 MiB > 32 MiB
    seqs = L.lpfa_seqs(1, rows, rows, rows, None, None)
    desc = L.lpfa_attn_desc(seqs, 1, 1, 128, 0.088, 1, 8.0, 1.0)
    st = L._bwd_noalloc(ctypes.byref(desc), *([None] * 17), None)
    assert st == L.LPFA_ERR_INVALID_ARG


@pytest.mark.gpu
def test_noalloc_matches_workspace_backward_twice(L):
    w = workloads.custom(seed=9, batch=2, seqlen=384, heads_q=4, heads_kv=2,
                         head_dim=128, causal=True)
    x = workloads.make_inputs(w)
    T = w.batch * w.seqlen
    q, k, v, do = (x[n].reshape(T, -1, w.head_dim).cuda() for n in ("q", "k", "v", "do"))
    seqs = L.dense_seqs(w.batch, w.seqlen)
    desc = L.attn_desc(seqs, w.heads_q, w.heads_kv, w.head_dim, w.causal,
                       w.softmax_scale)
    mq, mk, mv = L.quantize_forward_operands(q, k, v, seqs)
    o, lse, fws = L.attention_forward_mx(mq, mk, mv, desc)
    bq, bk, bv, bdo = L.quantize_backward_operands(q, k, v, do, seqs)
    ref = L.attention_backward_mx(bq, bk, bv, bdo, o, do, lse, desc)
    L.lpfa_check(ref[3])
    for _ in range(2):
        dq = torch.full_like(ref[0], float("nan"))
        dk = torch.full_like(ref[1], float("nan"))
        dv = torch.full_like(ref[2], float("nan"))
        L.lpfa_bwd_noalloc(desc, bq.data, bq.sf_mma, bq.sf_mma_t, bk.data,
                           bk.sf_mma, bk.sf_mma_t, bv.data, bv.sf_mma, bdo.data,
                           bdo.sf_mma, bdo.sf_mma_t, o, do, lse, dq, dk, dv)
        torch.cuda.synchronize()
        for got in (dq, dk, dv):
            assert torch.isfinite(got).all()
        assert torch.equal(dk, ref[1]) and torch.equal(dv, ref[2])
        assert _relfro(dq, ref[0]) <= DQ_TOL
    assert np.isfinite(float(dq.float().abs().max()))
