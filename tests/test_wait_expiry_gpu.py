"""Failure detection without a GPU fault: the forward's bounded waits.

lpfa_fwd_wait_expiry_selftest runs the forward kernel with its waits bounded
by a short limit and with the copy of each CTA's first key/value tile
withheld; the MMA warp's wait for that tile runs out.  The kernel must
record the error word (lpfa_check -> LPFA_ERR_TIMEOUT), raise its abort flag,
drain what it issued, free its tensor memory and return, leaving the context
usable: the next normal call on the same stream succeeds and matches the
oracle.  No wait is unbounded, nothing traps, no invalid address is touched.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads
from oracle import attention as A


@pytest.fixture(scope="module")
def L():
    from mxfp8_block_scaled_quantizer_gb300 import build
    build()
    from mxfp8_block_scaled_quantizer_gb300 import lpfa
    return lpfa


def test_selftest_rejects_bad_limits(L):
    """Host-side checks (no GPU needed): the limit must be 1 us .. 2 s."""
    seqs = L.lpfa_seqs(1, 128, 128, 128, None, None)
    desc = L.lpfa_attn_desc(seqs, 1, 1, 128, 0.088, 1, 8.0, 1.0)
    for limit in (0, 3000000):
        st = L._fwd_expiry(ctypes.byref(desc), *([None] * 9), 256, limit, None)
        assert st == L.LPFA_ERR_INVALID_ARG


@pytest.mark.gpu
@pytest.mark.parametrize("seqlen,causal", [(128, True), (512, False)])
def test_expired_wait_reports_timeout_and_context_survives(L, seqlen, causal):
    w = workloads.custom(seed=5, batch=1, seqlen=seqlen, heads_q=2, heads_kv=1,
                         head_dim=128, causal=causal)
    x = workloads.make_inputs(w, with_grad_out=False)
    T = seqlen
    q, k, v = (x[n].reshape(T, -1, w.head_dim).cuda() for n in ("q", "k", "v"))
    seqs = L.dense_seqs(1, seqlen)
    desc = L.attn_desc(seqs, w.heads_q, w.heads_kv, w.head_dim, causal, w.softmax_scale)
    mq, mk, mv = L.quantize_forward_operands(q, k, v, seqs)
    o = torch.empty((T, w.heads_q, w.head_dim), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.heads_q, T), dtype=torch.float32, device="cuda")
    ws = torch.empty(L.fwd_workspace_size(desc), dtype=torch.uint8, device="cuda")
    L.lpfa_fwd_wait_expiry_selftest(desc, mq.data, mq.sf_mma, mk.data, mk.sf_mma,
                                    mv.data, mv.sf_mma, o, lse, ws, 1000)
    assert L.check_status(ws) == L.LPFA_ERR_TIMEOUT
    # the same stream, a normal call: succeeds and is right
    o2, lse2, ws2 = L.attention_forward_mx(mq, mk, mv, desc)
    L.lpfa_check(ws2)
    ref = A.mx_attention_fwd(x["q"], x["k"], x["v"], causal=causal,
                             softmax_scale=w.softmax_scale, kv_tile=A.FWD_KEY_TILE)
    got = o2.float().cpu().numpy().reshape(ref["o"].shape)
    err = np.linalg.norm(got - ref["o"]) / np.linalg.norm(ref["o"])
    assert err <= 2e-2
    assert np.abs(lse2.cpu().numpy() - ref["lse"]).max() <= 1e-3
