"""MXFP8 codec and block quantizers, written from the format definitions (fp64).

TEST INFRASTRUCTURE ONLY.  This package is the CPU oracle that the CUDA path is
checked against.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import it; the
product path never does, and it shares no code with the CUDA sources.

What it follows
---------------
* "Low-Precision FlashAttention-4: End-to-End Block-Scaled Attention for NVIDIA
  Blackwell", section "Understanding OCP MXFP8 Microscaling on Blackwell": a
  block of 32 contiguous elements shares one 8-bit E8M0 scale
  s = 2^(E8M0 - 127); each element is an E4M3 value v_i, and the block decodes
  to s * v_i.
* "Low Precision Flash Attention 4: End-to-End Block-Scaled Attention for
  Blackwell", paragraphs 2-3: the backward pass quantizes in square [32, 32]
  blocks so that the E4M3 payload is transpose-invariant.
* The E4M3 element format itself (OCP 8-bit floating point, the "fn" variant
  the pages name): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits;
  exponent field 0 holds subnormals 2^-6 * m/8; S.1111.111 is NaN; there is no
  infinity; the largest finite magnitude is 448.

Readings where the pages are silent (each one is listed in the design notes):
* Scale exponent: e = floor(log2(amax)) - 8, i.e. the largest power of two that
  keeps amax * 2^-e below 2 * 2^8 (8 = the exponent of E4M3's largest binade),
  clamped to [-127, 127].  amax = 0 gives e = -127 (code 0) with zero
  payloads; a block holding Inf or NaN gives scale code 0xFF and payload 0x7F.
* Element rounding: round to nearest, ties to even; magnitudes above 448 are
  saturated to 448 (no NaN is produced from a finite input); the sign of zero
  is kept (-tiny encodes as 0x80).

* The other OCP MX element formats (E5M2, FP6 E3M2 / E2M3, FP4 E2M1) follow
  the same block rule with their own emax; see ``FORMATS``.

Parity pins for this module live in ``tests/test_oracle_mx.py``.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
E4M3_NAN = 0x7F
E8M0_NAN = 0xFF
E8M0_BIAS = 127
EMAX_E4M3 = 8


def _e4m3_value(code: int) -> float:
    sign = -1.0 if code & 0x80 else 1.0
    exp_field = (code >> 3) & 0xF
    mant = code & 0x7
    if exp_field == 0xF and mant == 0x7:
        return float("nan")
    if exp_field == 0:
        return sign * (mant / 8.0) * 2.0 ** -6
    return sign * (1.0 + mant / 8.0) * 2.0 ** (exp_field - 7)


#: decoded value of every E4M3 code 0..255 (fp64, exact)
E4M3_TABLE = np.array([_e4m3_value(c) for c in range(256)], dtype=np.float64)
# non-negative finite magnitudes, codes 0..126, strictly increasing
_POS = E4M3_TABLE[:127].copy()
assert np.all(np.diff(_POS) > 0)


def e4m3_decode(codes) -> np.ndarray:
    return E4M3_TABLE[np.asarray(codes, dtype=np.uint8)]


def e8m0_decode(codes) -> np.ndarray:
    c = np.asarray(codes, dtype=np.int64)
    out = np.ldexp(1.0, c - E8M0_BIAS)
    return np.where(c == E8M0_NAN, np.nan, out)


def e4m3_encode(x) -> np.ndarray:
    """Round fp64 values to E4M3 codes: RNE, saturate to 448, keep the sign."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    finite_or_inf = ~np.isnan(a)
    a_safe = np.where(finite_or_inf, a, 0.0)
    lo = np.searchsorted(_POS, a_safe, side="right") - 1   # largest <= a
    lo = np.clip(lo, 0, 126)
    hi = np.minimum(lo + 1, 126)
    mid = 0.5 * (_POS[lo] + _POS[hi])   # exact: both are short dyadics
    pick_hi = (hi != lo) & ((a_safe > mid) | ((a_safe == mid) & (hi % 2 == 0)))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    code = np.where(np.signbit(x), code | np.uint8(0x80), code).astype(np.uint8)
    code = np.where(finite_or_inf, code, np.uint8(E4M3_NAN)).astype(np.uint8)
    return code


# --------------------------------------------------- other MX element formats
# The OCP MX element formats besides E4M3 ("Low-Precision FlashAttention-4
# ...", which names MXFP8, MXFP6 and MXFP4 as the block-scaled MMA formats;
# "Low Precision Flash Attention 4 ...", paragraph 1), written from their
# definitions: sign, exponent field with bias, mantissa field; emax is the
# exponent of the largest finite binade, which the scale rule subtracts.
#   E5M2  5 exponent bits (bias 15), 2 mantissa bits, IEEE-like: exponent
#         field 31 holds Inf (mantissa 0) and NaN; max 57344; emax 15.
#   E3M2  (FP6) 3 / bias 3 / 2 bits, no Inf or NaN; max 28; emax 4.
#   E2M3  (FP6) 2 / bias 1 / 3 bits, no Inf or NaN; max 7.5; emax 2.
#   E2M1  (FP4) 2 / bias 1 / 1 bit, no Inf or NaN; max 6; emax 2.
# Codes hold one element each in the low bits of a byte (sign bit on top of
# the element's field).  A block holding Inf or NaN gets scale code 0xFF; its
# payload bytes are the format's NaN code (E5M2: 0x7F) or, for the formats
# without NaN, the largest positive code.
FORMATS = {
    # name: (exponent bits, mantissa bits, bias, emax, kind)
    "e4m3": (4, 3, 7, 8, "fn"),
    "e5m2": (5, 2, 15, 15, "ieee"),
    "e3m2": (3, 2, 3, 4, "finite"),
    "e2m3": (2, 3, 1, 2, "finite"),
    "e2m1": (2, 1, 1, 2, "finite"),
}


def _fmt_value(code: int, fmt: str) -> float:
    eb, mb, bias, _, kind = FORMATS[fmt]
    nbits = 1 + eb + mb
    sign = -1.0 if (code >> (nbits - 1)) & 1 else 1.0
    ef = (code >> mb) & ((1 << eb) - 1)
    m = code & ((1 << mb) - 1)
    if kind == "ieee" and ef == (1 << eb) - 1:
        return sign * float("inf") if m == 0 else float("nan")
    if kind == "fn" and ef == (1 << eb) - 1 and m == (1 << mb) - 1:
        return float("nan")
    if ef == 0:
        return sign * (m / 2.0 ** mb) * 2.0 ** (1 - bias)
    return sign * (1.0 + m / 2.0 ** mb) * 2.0 ** (ef - bias)


def fmt_table(fmt: str) -> np.ndarray:
    """Decoded value of every code of the format (fp64, exact)."""
    eb, mb, _, _, _ = FORMATS[fmt]
    return np.array([_fmt_value(c, fmt) for c in range(1 << (1 + eb + mb))], dtype=np.float64)


def fmt_nan_payload(fmt: str) -> int:
    """Payload byte of a block whose scale is NaN (0xFF)."""
    eb, mb, _, _, kind = FORMATS[fmt]
    if kind in ("fn", "ieee"):
        return 0x7F
    return (1 << (eb + mb)) - 1          # largest positive code


def fmt_encode(x, fmt: str) -> np.ndarray:
    """Round fp64 values to the format's codes: nearest, ties to the even
    code, magnitudes above the largest finite value saturate to it, the sign
    is kept (also of zero)."""
    if fmt == "e4m3":
        return e4m3_encode(x)
    eb, mb, _, _, _ = FORMATS[fmt]
    nbits = 1 + eb + mb
    table = fmt_table(fmt)
    npos = 1 << (nbits - 1)
    pos = table[:npos]
    finite = np.isfinite(pos)
    pos = pos[finite]                    # non-negative finite magnitudes, increasing
    last = len(pos) - 1
    assert np.all(np.diff(pos) > 0)
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    ok = ~np.isnan(a)
    a_safe = np.where(ok, a, 0.0)
    lo = np.clip(np.searchsorted(pos, a_safe, side="right") - 1, 0, last)
    hi = np.minimum(lo + 1, last)
    mid = 0.5 * (pos[lo] + pos[hi])
    pick_hi = (hi != lo) & ((a_safe > mid) | ((a_safe == mid) & (hi % 2 == 0)))
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    code = np.where(np.signbit(x), code | np.uint8(1 << (nbits - 1)), code).astype(np.uint8)
    return np.where(ok, code, np.uint8(fmt_nan_payload(fmt))).astype(np.uint8)


def scale_exponent(amax, emax: int = EMAX_E4M3) -> tuple:
    """(e, code) for block maxima amax >= 0: e = floor(log2 amax) - emax
    (8 for E4M3), clamped to [-127, 127]; amax == 0 -> e = -127; non-finite
    amax -> code 0xFF."""
    amax = np.asarray(amax, dtype=np.float64)
    finite = np.isfinite(amax)
    safe = np.where(finite & (amax > 0), amax, 1.0)
    _, fexp = np.frexp(safe)           # safe = f * 2^fexp, f in [0.5, 1)
    floor_log2 = fexp - 1
    e = floor_log2 - emax
    e = np.where(finite & (amax > 0), e, -E8M0_BIAS)
    e = np.clip(e, -127, 127)
    code = np.where(finite, e + E8M0_BIAS, E8M0_NAN).astype(np.uint8)
    return e.astype(np.int64), code


def _quantize_grouped(xg: np.ndarray, fmt: str = "e4m3"):
    """Quantize blocks laid out as the last axis of ``xg`` (shape [..., n]).
    Returns (payload codes [..., n], scale codes [...])."""
    amax = np.max(np.abs(xg), axis=-1) if xg.shape[-1] else np.zeros(xg.shape[:-1])
    e, code = scale_exponent(amax, FORMATS[fmt][3])
    scaled = np.ldexp(xg, -e[..., None])       # exact power-of-two scaling
    payload = fmt_encode(scaled, fmt)
    bad = code == E8M0_NAN
    if np.any(bad):
        payload = np.where(bad[..., None], np.uint8(fmt_nan_payload(fmt)), payload)
    return payload.astype(np.uint8), code


def quantize_1x32(x, fmt: str = "e4m3") -> tuple:
    """1x32 blocks along the last axis (length a multiple of 32).

    Returns (payload uint8 same shape, scale codes [..., n/32])."""
    x = np.asarray(x, dtype=np.float64)
    n = x.shape[-1]
    assert n % 32 == 0
    xg = x.reshape(*x.shape[:-1], n // 32, 32)
    payload, code = _quantize_grouped(xg, fmt)
    return payload.reshape(x.shape), code


def quantize_along_rows(x, block: int = 32, fmt: str = "e4m3") -> tuple:
    """Blocks of ``block`` consecutive rows (axis 0) per column, starting at
    row 0; the last block may be short (ragged sequence end).

    x: [R, ...]. Returns (payload [R, ...], scale codes [ceil(R/block), ...])."""
    x = np.asarray(x, dtype=np.float64)
    r = x.shape[0]
    nb = -(-r // block)
    pad = nb * block - r
    xp = np.concatenate([x, np.zeros((pad,) + x.shape[1:])], 0) if pad else x
    # zero padding cannot raise a block's amax; padded outputs are dropped
    xg = np.moveaxis(xp.reshape(nb, block, *x.shape[1:]), 1, -1)
    payload, code = _quantize_grouped(xg, fmt)
    payload = np.moveaxis(payload, -1, 1).reshape(nb * block, *x.shape[1:])[:r]
    return payload, code


def quantize_32x32(x, fmt: str = "e4m3") -> tuple:
    """Square 32x32 blocks over the first two axes of x [R, C, ...]; blocks
    start at (0, 0); the last row-block may be short, C must be a multiple
    of 32.  Returns (payload [R, C, ...], scales [ceil(R/32), C/32, ...])."""
    x = np.asarray(x, dtype=np.float64)
    r, c = x.shape[:2]
    assert c % 32 == 0
    nb = -(-r // 32)
    pad = nb * 32 - r
    xp = np.concatenate([x, np.zeros((pad,) + x.shape[1:])], 0) if pad else x
    rest = x.shape[2:]
    # [nb, 32, C/32, 32, ...] -> [nb, C/32, ..., 32*32]
    xg = xp.reshape(nb, 32, c // 32, 32, *rest)
    xg = np.moveaxis(xg, (1, 3), (-2, -1))
    xg = xg.reshape(nb, c // 32, *rest, 1024)
    payload, code = _quantize_grouped(xg, fmt)
    payload = payload.reshape(nb, c // 32, *rest, 32, 32)
    payload = np.moveaxis(payload, (-2, -1), (1, 3)).reshape(nb * 32, c, *rest)
    return payload[:r], code


def dequantize(payload, scale_codes, expand, fmt: str = "e4m3") -> np.ndarray:
    """Decode payload * 2^(scale - 127); ``expand`` maps the scale array to
    the payload's shape (e.g. a repeat along the block axis)."""
    vals = e4m3_decode(payload) if fmt == "e4m3" else fmt_table(fmt)[np.asarray(payload, np.uint8)]
    return vals * expand(e8m0_decode(scale_codes))


def dq_1x32(payload, sc, fmt: str = "e4m3"):
    return dequantize(payload, sc, lambda s: np.repeat(s, 32, axis=-1), fmt)


def dq_rows(payload, sc, block: int = 32):
    r = payload.shape[0]
    return dequantize(payload, sc,
                      lambda s: np.repeat(s, block, axis=0)[:r])


def dq_32x32(payload, sc):
    r = payload.shape[0]
    return dequantize(payload, sc,
                      lambda s: np.repeat(np.repeat(s, 32, axis=0), 32, axis=1)[:r])


def fake_quant_1x32(x):
    return dq_1x32(*quantize_1x32(x))


def fake_quant_rows(x):
    return dq_rows(*quantize_along_rows(x))


def fake_quant_32x32(x):
    return dq_32x32(*quantize_32x32(x))


def mx_gemm(a_payload, a_sc, b_payload, b_sc, a_fmt: str = "e4m3",
            b_fmt: str = "e4m3") -> np.ndarray:
    """D = A @ B^T with A [M, K], B [N, K] both 1x32-blocked along K (the
    block-scaled MMA's contraction), each in its own element format.  Every
    product of two decoded operands is exact in fp64, so this is the dense
    GEMM of the dequantized operands."""
    return dq_1x32(a_payload, a_sc, a_fmt) @ dq_1x32(b_payload, b_sc, b_fmt).T


# --------------------------------------------------------------- NVFP4
# NVFP4 ("Low Precision Flash Attention 4 ...", paragraph 2, names it among
# the formats the block-scaled MMA takes; the pages give no rule).  Reading:
# blocks of 16 consecutive elements along the contraction, E2M1 elements
# (largest magnitude 6), one positive E4M3 scale per block, no second-level
# per-tensor scale.  In fp32, as the kernel computes it:
#   s = E4M3(amax / 6)                 round to nearest even, saturating
#   element = E2M1(x / s)              round to nearest even, saturating at 6
# A block with amax = 0 (or a scale that rounds to 0) has scale code 0 and
# zero payloads.  The divisions are single fp32 divisions, so their rounding
# is part of the definition.
NVFP4_BLOCK = 16


def quantize_nvfp4(x) -> tuple:
    """16-element blocks along the last axis.  Returns (E2M1 codes, one per
    byte [..., n], E4M3 scale codes [..., n/16])."""
    x32 = np.asarray(x, dtype=np.float32)
    n = x32.shape[-1]
    assert n % NVFP4_BLOCK == 0
    xg = x32.reshape(*x32.shape[:-1], n // NVFP4_BLOCK, NVFP4_BLOCK)
    amax = np.max(np.abs(xg), axis=-1)
    s32 = (amax / np.float32(6.0)).astype(np.float32)     # one fp32 division
    s_code = e4m3_encode(s32.astype(np.float64))
    s = e4m3_decode(s_code).astype(np.float32)
    safe = np.where(s > 0, s, np.float32(1.0))
    y = (xg / safe[..., None]).astype(np.float32)         # one fp32 division
    codes = fmt_encode(y.astype(np.float64), "e2m1")
    codes = np.where((s > 0)[..., None], codes, np.uint8(0)).astype(np.uint8)
    s_code = np.where(s > 0, s_code, np.uint8(0)).astype(np.uint8)
    return codes.reshape(x32.shape), s_code


def dq_nvfp4(codes, s_code):
    vals = fmt_table("e2m1")[np.asarray(codes, np.uint8)]
    s = e4m3_decode(s_code)
    return vals * np.repeat(s, NVFP4_BLOCK, axis=-1)


def fp4_gemm(a_codes, a_sc, b_codes, b_sc, scale: str) -> np.ndarray:
    """D = A @ B^T for E2M1 operands with 32-element E8M0 blocks
    (scale='mx') or 16-element E4M3 blocks (scale='nv'); every product of two
    decoded operands is exact in fp64."""
    if scale == "mx":
        return dq_1x32(a_codes, a_sc, "e2m1") @ dq_1x32(b_codes, b_sc, "e2m1").T
    return dq_nvfp4(a_codes, a_sc) @ dq_nvfp4(b_codes, b_sc).T
