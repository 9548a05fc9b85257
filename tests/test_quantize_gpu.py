"""Quantizer parity on the GPU: E4M3 payloads and E8M0 scales (compact and
both tensor-core arrangements) bit-exact against the oracle, on every
workload's tensors (sampled tokens for the two largest) and on edge cases."""
import numpy as np
import pytest
import torch

import workloads
from oracle import layouts

pytestmark = pytest.mark.gpu

BLOCKS = {"1x32": 0, "32x1": 1, "32x32": 2}


@pytest.fixture(scope="module")
def L():
    from mxfp8_block_scaled_quantizer_gb300 import build
    build()
    from mxfp8_block_scaled_quantizer_gb300 import lpfa
    assert lpfa.lpfa_device_supported()
    return lpfa


def _gpu_quant(L, x_tok, cu, block):
    x = x_tok.cuda().contiguous()
    if cu is None:
        seqs = L.dense_seqs(1, x.shape[0])
    else:
        seqs = L.varlen_seqs(torch.as_tensor(cu, dtype=torch.int32))
    m = L.mx_quantize(x, BLOCKS[block], seqs)
    torch.cuda.synchronize()
    return {k: (None if getattr(m, k) is None else getattr(m, k).cpu().numpy())
            for k in ("data", "sf", "sf_mma", "sf_mma_t")}


def _compare(got, want, tag):
    assert np.array_equal(got["data"], want["payload"]), f"{tag}: payload"
    assert np.array_equal(got["sf"], want["sf"]), f"{tag}: compact scales"
    assert np.array_equal(got["sf_mma"], want["sf_mma"]), f"{tag}: mma scales"
    if want["sf_mma_t"] is not None:
        assert np.array_equal(got["sf_mma_t"], want["sf_mma_t"]), f"{tag}: mma_t"


def _check(L, x_tok, cu, block, tag):
    got = _gpu_quant(L, x_tok, cu, block)
    cu_o = np.array([0, x_tok.shape[0]]) if cu is None else np.asarray(cu)
    want = layouts.oracle_quantize(x_tok.float().numpy(), cu_o, block)
    _compare(got, want, tag)


@pytest.mark.parametrize("block", list(BLOCKS))
@pytest.mark.parametrize("name", ["tiny", "outlier"])
def test_quantizer_small_workloads_full(L, name, block):
    w = workloads.get_config(name)
    x = workloads.make_inputs(w)
    for t in ("q", "k", "v", "do"):
        xt = x[t].reshape(-1, *x[t].shape[2:])
        cu = np.arange(w.batch + 1) * w.seqlen
        _check(L, xt, cu, block, f"{name}.{t}")


@pytest.mark.parametrize("block", list(BLOCKS))
def test_quantizer_varlen_sampled_sequences(L, block):
    """Jagged inputs: a few whole sequences (shortest, longest, two more)
    packed unpadded with their own cu_seqlens."""
    w = workloads.get_config("varlen")
    x = workloads.make_inputs(w)
    lens = x["lengths"].numpy()
    cu = x["cu_seqlens"].numpy()
    pick = sorted({int(lens.argmin()), int(lens.argmax()), 0, 17})
    parts = [x["k"][cu[s]:cu[s + 1]] for s in pick]
    sub_cu = np.concatenate([[0], np.cumsum([p.shape[0] for p in parts])])
    _check(L, torch.cat(parts, 0), sub_cu, block, "varlen.k")


@pytest.mark.parametrize("block", list(BLOCKS))
@pytest.mark.parametrize("name", ["llm", "gqa_long"])
def test_quantizer_large_workloads_sampled(L, name, block):
    """Full-size tensors quantized on the GPU in the bench's launch
    configuration; token windows compared with the oracle."""
    w = workloads.get_config(name)
    torch.manual_seed(0)
    x = workloads.make_inputs(w, with_grad_out=False)["q"]
    B, S, H, D = x.shape
    xt = x.reshape(B * S, H, D)
    seqs = L.dense_seqs(B, S)
    m = L.mx_quantize(xt.cuda(), BLOCKS[block], seqs)
    torch.cuda.synchronize()
    for start in (0, S - 256, (B - 1) * S + 4096):
        win = xt[start:start + 256]
        want = layouts.oracle_quantize(win.float().numpy(), np.array([0, 256]), block)
        got = {"data": m.data[start:start + 256].cpu().numpy()}
        if block == "1x32":
            got["sf"] = m.sf[start:start + 256].cpu().numpy()
        else:
            got["sf"] = m.sf[start // 32:(start + 256) // 32].cpu().numpy()
        got["sf_mma"] = m.sf_mma[start // 128:(start + 256) // 128].cpu().numpy()
        got["sf_mma_t"] = None if m.sf_mma_t is None else \
            m.sf_mma_t[start // 128:(start + 256) // 128].cpu().numpy()
        _compare(got, want, f"{name}@{start}")


def _edge_tensor():
    """Special values: zeros, bf16 subnormals, huge values, exact rounding
    midpoints after scaling, negative zero, saturating elements."""
    rng = np.random.default_rng(7)
    T, H, D = 96, 2, 64
    x = rng.standard_normal((T, H, D)).astype(np.float32)
    x[0:32, 0, 0:32] = 0.0                                  # all-zero block
    x[32, 0, :] = np.float32(2.0 ** -130)                   # bf16 subnormals
    x[33, 0, :] = -np.float32(2.0 ** -133)
    x[34, 1, :] = np.float32(3.0e38)                        # near bf16 max
    x[35, 1, 0:32] = np.array([2.375 * 2 ** k for k in range(-16, 16)], np.float32)
    x[36, 0, 0:32] = -0.0
    x[36, 0, 0] = 1.0
    x[37, 1, 32:64] = np.linspace(-448, 448, 32).astype(np.float32)
    x[38, 0, 0:32] = np.float32(1.0)
    x[38, 0, 5] = np.float32(1.9999)                        # block max rounds
    return torch.from_numpy(x).to(torch.bfloat16)


@pytest.mark.parametrize("block", list(BLOCKS))
def test_quantizer_edge_values(L, block):
    x = _edge_tensor()
    _check(L, x, np.array([0, 96]), block, "edge")
    # ragged sequences, lengths not multiples of 32 or 128
    _check(L, x, np.array([0, 5, 40, 41, 96]), block, "edge-ragged")


def test_quantizer_nonfinite_blocks(L):
    x = torch.randn(64, 1, 128).to(torch.bfloat16)
    x[3, 0, 7] = float("inf")
    x[40, 0, 100] = float("nan")
    for block in BLOCKS:
        _check(L, x, np.array([0, 64]), block, f"nonfinite-{block}")


def test_quantizer_empty_and_single_token(L):
    x = torch.randn(1, 3, 128).to(torch.bfloat16)
    for block in BLOCKS:
        _check(L, x, np.array([0, 1]), block, f"single-{block}")


FORMATS = {"e5m2": 1, "e3m2": 2, "e2m3": 3, "e2m1": 4}


@pytest.mark.parametrize("fmt", list(FORMATS))
@pytest.mark.parametrize("block", list(BLOCKS))
def test_quantizer_other_element_formats(L, fmt, block):
    """E5M2, FP6 (E3M2, E2M3) and FP4 (E2M1) payloads and scales bit-exact
    on the outlier workload's Q (wide dynamic range), a ragged packed batch
    and the edge tensor (zeros, Inf/NaN blocks, saturation)."""
    w = workloads.get_config("outlier")
    x = workloads.make_inputs(w)
    edge = _edge_tensor().clone()
    edge[40, 0, 3] = float("nan")
    edge[41, 1, 40] = float("inf")
    cases = [(x["q"].reshape(-1, *x["q"].shape[2:])[:300], [0, 300]), (edge, None)]
    for i, (xt, cu) in enumerate(cases):
        xc = xt.cuda().contiguous()
        seqs = L.dense_seqs(1, xc.shape[0]) if cu is None else \
            L.varlen_seqs(torch.as_tensor(cu, dtype=torch.int32))
        m = L.mx_quantize(xc, BLOCKS[block], seqs, fmt=FORMATS[fmt])
        torch.cuda.synchronize()
        got = {k: (None if getattr(m, k) is None else getattr(m, k).cpu().numpy())
               for k in ("data", "sf", "sf_mma", "sf_mma_t")}
        cu_o = np.array([0, xt.shape[0]]) if cu is None else np.asarray(cu)
        want = layouts.oracle_quantize(xt.float().numpy(), cu_o, block, fmt)
        _compare(got, want, f"{fmt}.{block}.{i}")
