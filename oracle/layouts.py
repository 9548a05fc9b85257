"""Scale-factor arrangements used by the quantizer's outputs (test side).

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Two arrangements exist for every quantized operand:

* compact: one E8M0 byte per block, indexed naturally
    - 1x32 along head_dim:      [T, H, D/32]
    - 32 along tokens:          [Tp/32, H, D]
    - 32x32 (tokens, head_dim): [Tp/32, H, D/32]
  where token-blocked arrays index tokens in the padded scale-row space below.
* MMA-ready: the layout the tensor core reads scale factors in, per 128-row
  operand tile: 128 operand rows x 4 contraction blocks (128 contraction
  elements) = 512 bytes, where operand row r and contraction block kb sit at
  byte (r % 32) * 16 + (r // 32) * 4 + kb.  Tiles are stored [Tp/128, H, 512].
  "Operand rows" are tokens for K-major use (contraction over head_dim) and
  head_dim channels for MN-major use (contraction over tokens).

``gemm_operand_mma`` / ``gemm_quantize`` give the same arrangements for a
GEMM result quantized as the next GEMM's operand (the fused GEMM+Quantize
producer of "Low Precision Flash Attention 4", paragraph 2): codes are decided
on the kernel's own fp32 result, so the comparison with the fused output is
exact.

Padded scale rows (the jagged module of "Low Precision Flash Attention 4",
paragraph 2): FP8 data stays at unpadded token positions; scale rows of
sequence s start at the 128-aligned row sf_start[s] = sum_{t<s} ceil(L_t/128)
* 128, so every 128-token tile of every sequence owns whole 512-byte scale
tiles.  Unused bytes are zero.
"""
from __future__ import annotations

import numpy as np


def sf_row_starts(cu_seqlens) -> np.ndarray:
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    lens = np.diff(cu)
    padded = -(-lens // 128) * 128
    return np.concatenate([[0], np.cumsum(padded)]).astype(np.int64)


def atom_offset(r, kb):
    r = np.asarray(r); kb = np.asarray(kb)
    return (r % 32) * 16 + (r // 32) * 4 + kb


def _token_rows(cu_seqlens):
    """(sequence id, padded scale row) of every token."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    lens = np.diff(cu)
    sfs = sf_row_starts(cu)
    seq = np.repeat(np.arange(len(lens)), lens)
    i = np.arange(cu[-1]) - cu[seq]
    return seq, sfs[seq] + i


def mma_from_row_blocks(row_sc, cu_seqlens):
    """K-major arrangement from per-token scales row_sc [T, H, nkb]
    (nkb = D/32 <= 4).  Returns uint8 [Tp/128, H, 512]."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    sfs = sf_row_starts(cu)
    T, H, nkb = row_sc.shape
    _, pr = _token_rows(cu)
    out = np.zeros((sfs[-1] // 128, 512, H), dtype=np.uint8)
    for kb in range(nkb):
        out[pr // 128, atom_offset(pr % 128, kb), :] = row_sc[:, :, kb]
    return np.ascontiguousarray(np.moveaxis(out, 2, 1))


def mma_from_token_blocks(col_sc, D):
    """MN-major arrangement from 32-token-block scales col_sc [Tp/32, H, D]
    (one scale per (token block, head_dim channel)).  Operand rows are the
    head_dim channels, contraction blocks the 4 token blocks of a tile."""
    nblk, H, d = col_sc.shape
    assert d == D
    out = np.zeros((-(-nblk // 4), 512, H), dtype=np.uint8)
    tb, ch = np.meshgrid(np.arange(nblk), np.arange(D), indexing="ij")
    out[tb // 4, atom_offset(ch, tb % 4), :] = col_sc[tb, :, ch]
    return np.ascontiguousarray(np.moveaxis(out, 2, 1))


def square_to_row(sq_sc, cu_seqlens):
    """Per-token view [T, H, D/32] of square scales [Tp/32, H, D/32]."""
    _, pr = _token_rows(cu_seqlens)
    return sq_sc[pr // 32]


def square_to_col(sq_sc, D):
    """Per-(token block, channel) view [Tp/32, H, D] of square scales."""
    return np.repeat(sq_sc, 32, axis=2)[:, :, :D]


def oracle_quantize(x, cu_seqlens, block, fmt="e4m3"):
    """Oracle quantization of a token-major tensor x [T, H, D] with the
    library's output layouts.  block: "1x32", "32x1" or "32x32"; fmt: the
    element format (``mx.FORMATS``).
    Returns dict(payload [T,H,D] uint8, sf (compact), sf_mma, sf_mma_t)."""
    from . import mx
    x = np.asarray(x, dtype=np.float64)
    T, H, D = x.shape
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    sfs = sf_row_starts(cu)
    out = {"sf_mma_t": None}
    if block == "1x32":
        p, sc = mx.quantize_1x32(x, fmt)
        out.update(payload=p, sf=sc, sf_mma=mma_from_row_blocks(sc, cu))
        return out
    payload = np.zeros((T, H, D), dtype=np.uint8)
    if block == "32x1":
        sc = np.zeros((sfs[-1] // 32, H, D), dtype=np.uint8)
        for s in range(len(cu) - 1):
            a, b = cu[s], cu[s + 1]
            if b == a:
                continue
            p, c = mx.quantize_along_rows(x[a:b], fmt=fmt)
            payload[a:b] = p
            sc[sfs[s] // 32: sfs[s] // 32 + c.shape[0]] = c
        out.update(payload=payload, sf=sc, sf_mma=mma_from_token_blocks(sc, D))
        return out
    assert block == "32x32"
    sc = np.zeros((sfs[-1] // 32, H, D // 32), dtype=np.uint8)
    for s in range(len(cu) - 1):
        a, b = cu[s], cu[s + 1]
        if b == a:
            continue
        p, c = mx.quantize_32x32(np.moveaxis(x[a:b], 2, 1), fmt)   # [L, D, H]
        payload[a:b] = np.moveaxis(p, 1, 2)
        sc[sfs[s] // 32: sfs[s] // 32 + c.shape[0]] = np.moveaxis(c, 1, 2)
    row = square_to_row(sc, cu)
    out.update(payload=payload, sf=sc, sf_mma=mma_from_row_blocks(row, cu),
               sf_mma_t=mma_from_token_blocks(square_to_col(sc, D), D))
    return out


# ------------------------------------------------------------------ GEMM outputs
def gemm_operand_mma(sc):
    """Tensor-core arrangement of a GEMM operand's scales: sc [R, C/32]
    (one code per row and 32-element block along the contraction) ->
    uint8 [R/128][C/128][512], tile (i, j) holding rows 128 i .. and
    contraction blocks 4 j .. 4 j + 3 at atom_offset(row % 128, block % 4)."""
    R, nb = sc.shape
    out = np.zeros((R // 128, -(-nb // 4), 512), dtype=np.uint8)
    r, kb = np.meshgrid(np.arange(R), np.arange(nb), indexing="ij")
    out[r // 128, kb // 4, atom_offset(r % 128, kb % 4)] = sc[r, kb]
    return out


def gemm_quantize(d, block):
    """Oracle of the quantizing GEMM epilogue: the fp32 result d [M, N]
    quantized in 1x32 blocks along N, or in 32x32 blocks.  Returns dict(
    payload [M, N], sf (compact: [M, N/32] or [M/32, N/32]), sf_mma (rows =
    M, contraction over N: [M/128][N/128][512]) and, for 32x32, sf_mma_t
    (rows = N, contraction over M: [N/128][M/128][512]))."""
    from . import mx
    d = np.asarray(d, dtype=np.float64)
    if block == "1x32":
        p, sc = mx.quantize_1x32(d)
        return {"payload": p, "sf": sc, "sf_mma": gemm_operand_mma(sc), "sf_mma_t": None}
    assert block == "32x32"
    p, sc = mx.quantize_32x32(d)
    return {"payload": p, "sf": sc,
            "sf_mma": gemm_operand_mma(np.repeat(sc, 32, axis=0)),
            "sf_mma_t": gemm_operand_mma(np.repeat(sc.T, 32, axis=0))}


# ------------------------------------------------------ MMA operand bytes
def mma_operand_bytes(codes, fmt):
    """The byte layout block-scaled MMAs read for an operand of element
    format ``fmt``: codes [R, C] (one code per byte, C a multiple of 16) ->
    bytes [R, C].  E4M3 / E5M2: unchanged.  FP6 (e3m2, e2m3) and FP4 (e2m1):
    every 16 consecutive codes of a row form one 16-byte group holding their
    bits as a little-endian stream (code j at bits b*j .. b*j + b - 1 of the
    group, b = 6 or 4) followed by zero bytes."""
    codes = np.asarray(codes, dtype=np.uint8)
    if fmt in ("e4m3", "e5m2"):
        return codes.copy()
    bits = {"e3m2": 6, "e2m3": 6, "e2m1": 4}[fmt]
    R, C = codes.shape
    assert C % 16 == 0
    out = np.zeros((R, C), dtype=np.uint8)
    mask = (1 << bits) - 1
    for g in range(C // 16):
        stream = np.zeros(R, dtype=object)
        for j in range(16):
            stream = stream + ((codes[:, 16 * g + j].astype(object) & mask) << (bits * j))
        for byte in range(bits * 2):           # 16 codes * bits / 8
            out[:, 16 * g + byte] = np.array([(int(v) >> (8 * byte)) & 0xFF for v in stream],
                                             dtype=np.uint8)
    return out


def fp4_dense_bytes(codes):
    """Dense FP4 operand bytes: codes [R, C] (one E2M1 code per byte, C
    even) -> [R, C/2], code 2i in the low nibble and code 2i + 1 in the high
    nibble of byte i."""
    c = np.asarray(codes, dtype=np.uint8) & 0xF
    return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)
