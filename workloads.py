"""Seeded synthetic inputs for MXFP8 block-scaled attention.

This module holds the input recipes only: it draws random numbers and shapes
tensors, and contains none of the method's arithmetic (no quantization, no
attention).  It is the one module that both the CPU oracle's tests and the CUDA
path's tests, ``bench.py`` and ``__graft_entry__`` use, so that both sides see
identical bf16 bytes.

Recipe (every config): a CPU ``torch.Generator`` seeded with the config's seed
draws fp32 N(0, 1) tensors in the order Q, K, V, dO; each draw is reshaped,
structured as the config says, then cast to bf16 (round to nearest even).

The five workloads follow the shapes the pages use (batch 8, 8192 tokens,
32 heads, head_dim 128, causal, from the PyTorch invocation example of
"Low-Precision FlashAttention-4: End-to-End Block-Scaled Attention for NVIDIA
Blackwell"), plus a tiny case, an outlier case, a long-context GQA case and a
jagged (varlen) case.  The pages' own "LLM shapes" and "internal shapes" are not
given; these synthetic inputs stand in for them.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

__all__ = ["Workload", "CONFIGS", "get_config", "make_inputs", "attn_flops"]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int                  # sequences (dense: B)
    seqlen: int                 # dense: S; varlen: 0 (lengths are drawn)
    heads_q: int
    heads_kv: int
    head_dim: int
    causal: bool
    seed: int
    outlier_channels: tuple = ()   # head_dim channels scaled in Q and K
    outlier_gain: float = 1.0
    token_lognormal_sigma: float = 0.0   # per-token norm factor exp(sigma*z)
    varlen: bool = False
    varlen_min: int = 0
    varlen_max: int = 0

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)


CONFIGS = {
    "tiny": Workload("tiny", batch=1, seqlen=256, heads_q=2, heads_kv=2,
                     head_dim=64, causal=False, seed=0),
    "outlier": Workload("outlier", batch=2, seqlen=2048, heads_q=16,
                        heads_kv=16, head_dim=128, causal=True, seed=1,
                        outlier_channels=(1, 9, 17, 25), outlier_gain=20.0),
    "llm": Workload("llm", batch=8, seqlen=8192, heads_q=32, heads_kv=32,
                    head_dim=128, causal=True, seed=2),
    "gqa_long": Workload("gqa_long", batch=1, seqlen=32768, heads_q=64,
                         heads_kv=8, head_dim=128, causal=True, seed=3,
                         token_lognormal_sigma=0.5),
    "varlen": Workload("varlen", batch=64, seqlen=0, heads_q=16, heads_kv=16,
                       head_dim=128, causal=False, seed=4, varlen=True,
                       varlen_min=128, varlen_max=4096),
}


def get_config(name: str) -> Workload:
    return CONFIGS[name]


def custom(**kw) -> Workload:
    """A workload with explicit fields (for edge-case tests)."""
    base = dict(name="custom", batch=1, seqlen=128, heads_q=1, heads_kv=1,
                head_dim=128, causal=False, seed=0)
    base.update(kw)
    return Workload(**base)


def seqlens(w: Workload, gen: Optional[torch.Generator] = None) -> torch.Tensor:
    """Sequence lengths (int64, CPU).  Varlen lengths are uniform integers in
    [varlen_min, varlen_max], drawn first from the config's generator."""
    if not w.varlen:
        return torch.full((w.batch,), w.seqlen, dtype=torch.int64)
    if gen is None:
        gen = torch.Generator("cpu").manual_seed(w.seed)
    return torch.randint(w.varlen_min, w.varlen_max + 1, (w.batch,),
                         generator=gen)


def cu_seqlens_of(lengths: torch.Tensor) -> torch.Tensor:
    cu = torch.zeros(lengths.numel() + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(lengths, 0).to(torch.int32)
    return cu


def make_inputs(w: Workload, with_grad_out: bool = True) -> dict:
    """Draw Q, K, V (and dO) as bf16 CPU tensors.

    Dense configs give [B, S, H, D] (BSHD); varlen gives packed [T, H, D] with
    ``cu_seqlens`` (int32, length batch+1).
    """
    gen = torch.Generator("cpu").manual_seed(w.seed)
    lengths = seqlens(w, gen)
    if w.varlen:
        total = int(lengths.sum())
        lead = (total,)
    else:
        total = w.batch * w.seqlen
        lead = (w.batch, w.seqlen)

    def draw(heads: int, outliers: bool) -> torch.Tensor:
        x = torch.randn(*lead, heads, w.head_dim, generator=gen,
                        dtype=torch.float32)
        if outliers and w.outlier_channels:
            idx = torch.tensor(w.outlier_channels, dtype=torch.int64)
            x[..., idx] *= w.outlier_gain
        if w.token_lognormal_sigma:
            z = torch.randn(*lead, generator=gen, dtype=torch.float32)
            x *= torch.exp(w.token_lognormal_sigma * z)[..., None, None]
        return x.to(torch.bfloat16)

    out = {
        "q": draw(w.heads_q, True),
        "k": draw(w.heads_kv, True),
        "v": draw(w.heads_kv, False),
    }
    if with_grad_out:
        out["do"] = draw(w.heads_q, False)
    out["lengths"] = lengths
    out["cu_seqlens"] = cu_seqlens_of(lengths)
    out["total"] = total
    return out


def attn_flops(w: Workload, lengths: Optional[torch.Tensor] = None) -> tuple:
    """(forward, backward) FLOPs: 4*H*Sq*Sk*D and 10*H*Sq*Sk*D per sequence,
    halved for causal, with H the number of query heads."""
    if lengths is None:
        lengths = seqlens(w)
    sq2 = float((lengths.to(torch.float64) ** 2).sum())
    f = 0.5 if w.causal else 1.0
    fwd = 4.0 * w.heads_q * sq2 * w.head_dim * f
    bwd = 10.0 * w.heads_q * sq2 * w.head_dim * f
    return fwd, bwd


# --------------------------------------------------------------- GEMM-Norm
# The jagged GEMM-Norm backward's inputs: a jagged batch of token rows (the
# sequences concatenated, lengths uniform in [len_min, len_max]) through a
# hidden x hidden projection.  The pages give no shape for it; these stand in.
GEMM_NORM = {"batch": 16, "len_min": 128, "len_max": 8192, "hidden": 4096, "seed": 5}


def gemm_norm_lengths(batch: int, len_min: int, len_max: int, seed: int) -> torch.Tensor:
    gen = torch.Generator("cpu").manual_seed(seed)
    return torch.randint(len_min, len_max + 1, (batch,), generator=gen)


def gemm_norm_inputs(T: int, N: int, K: int, seed: int) -> dict:
    """X [T, K] ~ N(0, 1), W [N, K] ~ N(0, 1/K), gamma [N] ~ 1 + 0.1 N(0, 1),
    dZ [T, N] ~ N(0, 1), drawn in that order from one seeded CPU generator and
    cast to bf16."""
    gen = torch.Generator("cpu").manual_seed(seed)
    x = torch.randn(T, K, generator=gen)
    w = torch.randn(N, K, generator=gen) / math.sqrt(K)
    gamma = 1.0 + 0.1 * torch.randn(N, generator=gen)
    dz = torch.randn(T, N, generator=gen)
    return {"x": x.to(torch.bfloat16), "w": w.to(torch.bfloat16),
            "gamma": gamma.to(torch.bfloat16), "dz": dz.to(torch.bfloat16)}
