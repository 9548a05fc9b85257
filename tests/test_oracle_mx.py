"""Pins for the oracle's MX codec and quantizers (CPU only).

Each test ties the oracle to something other than itself: torch's independent
fp8 decoders, brute-force nearest search, closed forms of the scale rule, the
transpose invariance of square blocks stated in "Low Precision Flash
Attention 4: End-to-End Block-Scaled Attention for Blackwell" (paragraph 3),
and the decomposition x = 2^(E8M0-127) * v from "Low-Precision
FlashAttention-4 ..." ("Understanding OCP MXFP8 Microscaling on Blackwell").
"""
import os

import numpy as np
import pytest
import torch

from oracle import mx, layouts

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- decode pins
def test_e4m3_decode_matches_torch_all_codes():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn)
    ref = ref.to(torch.float64).numpy()
    ours = mx.E4M3_TABLE
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert nan.sum() == 2          # 0x7F and 0xFF only


def test_e4m3_landmarks():
    assert mx.E4M3_TABLE[0x7E] == 448.0          # largest finite
    assert mx.E4M3_TABLE[0x01] == 2.0 ** -9      # smallest subnormal
    assert mx.E4M3_TABLE[0x08] == 2.0 ** -6      # smallest normal
    assert mx.E4M3_TABLE[0x38] == 1.0
    assert mx.E4M3_TABLE[0x80] == 0.0 and np.signbit(mx.E4M3_TABLE[0x80])


def test_e8m0_decode_matches_torch_and_golden():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu)
    ref = ref.to(torch.float64).numpy()
    ours = mx.e8m0_decode(np.arange(256))
    assert np.isnan(ours[255]) and np.isnan(ref[255])
    assert np.array_equal(ours[:255], ref[:255])
    # s = 2^(E8M0 - 127), sampled codes in tests/golden/e8m0_scale_codes.txt
    rows = np.loadtxt(os.path.join(GOLDEN, "e8m0_scale_codes.txt"),
                      comments="#")
    for code, log2s in rows:
        assert mx.e8m0_decode(int(code)) == 2.0 ** log2s


# ---------------------------------------------------------------- encode pins
def _brute_nearest(a):
    """Nearest finite E4M3 code by exhaustive search, ties to even code,
    saturating; sign applied separately."""
    mags = mx.E4M3_TABLE[:127]
    out = []
    for v in a:
        m = min(abs(v), 448.0)
        d = np.abs(mags - m)
        best = np.flatnonzero(d == d.min())
        code = best[0] if len(best) == 1 else best[best % 2 == 0][0]
        out.append(code | (0x80 if np.signbit(v) else 0))
    return np.array(out, dtype=np.uint8)


def test_e4m3_encode_exact_values_roundtrip():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)],
                     dtype=np.uint8)
    assert np.array_equal(mx.e4m3_encode(mx.E4M3_TABLE[codes]), codes)


def test_e4m3_encode_midpoints_go_to_even():
    mags = mx.E4M3_TABLE[:127]
    mids = 0.5 * (mags[:-1] + mags[1:])
    got = mx.e4m3_encode(mids)
    lo = np.arange(126)
    expect = np.where(lo % 2 == 0, lo, lo + 1)
    assert np.array_equal(got, expect.astype(np.uint8))
    assert np.array_equal(mx.e4m3_encode(-mids), (expect | 0x80).astype(np.uint8))


def test_e4m3_encode_vs_brute_force_random(rng):
    x = np.concatenate([
        rng.standard_normal(4000) * 50,
        rng.standard_normal(2000) * 1e-2,
        rng.uniform(-600, 600, 2000),
        np.ldexp(rng.uniform(0.5, 1, 500), rng.integers(-14, 10, 500)),
    ])
    assert np.array_equal(mx.e4m3_encode(x), _brute_nearest(x))


def test_e4m3_encode_vs_torch_in_range(rng):
    # torch rounds to nearest even too; it only differs above 464 (NaN).
    x = rng.uniform(-464, 464, 20000)
    x = x[np.abs(x) < 464]
    ref = torch.from_numpy(x).to(torch.float32).to(torch.float8_e4m3fn)
    ref = ref.view(torch.uint8).numpy()
    # compare on fp32-representable inputs (torch converts from fp32)
    x32 = x.astype(np.float32).astype(np.float64)
    assert np.array_equal(mx.e4m3_encode(x32), ref)


def test_e4m3_saturation_and_signed_zero():
    assert mx.e4m3_encode(np.array([449.0, 463.9, 464.0, 500.0, 1e30, np.inf])).tolist() == [126] * 6
    assert mx.e4m3_encode(np.array([-1e30]))[0] == 0xFE
    assert mx.e4m3_encode(np.array([-1e-30]))[0] == 0x80
    assert mx.e4m3_encode(np.array([1e-30]))[0] == 0x00
    assert mx.e4m3_encode(np.array([2.0 ** -10]))[0] == 0x00   # tie -> even (0)
    assert mx.e4m3_encode(np.array([3 * 2.0 ** -11]))[0] == 0x01
    assert mx.e4m3_encode(np.array([np.nan]))[0] == 0x7F


# ------------------------------------------------------------ scale rule pins
@pytest.mark.parametrize("k", list(range(-20, 20)))
def test_scale_rule_closed_form(k):
    """amax in [2^k, 2^(k+1)) -> code k - 8 + 127."""
    for frac in (1.0, 1.25, 1.999999):
        amax = frac * 2.0 ** k
        e, code = mx.scale_exponent(np.array([amax]))
        assert e[0] == k - 8 and code[0] == k - 8 + 127


def test_scale_rule_edges():
    e, code = mx.scale_exponent(np.array([0.0, np.inf, np.nan, 2.0 ** -140,
                                          2.0 ** 135, 448.0, 1.0]))
    assert code.tolist() == [0, 255, 255, 0, 254, 127, 119]


def test_block_max_roundtrip_property(rng):
    """The block max decodes within 2^-4 relative, or saturates at 448*2^e."""
    x = rng.standard_normal((500, 32)) * np.exp(rng.uniform(-10, 10, (500, 1)))
    p, sc = mx.quantize_1x32(x)
    amax = np.abs(x).max(axis=1)
    i = np.abs(x).argmax(axis=1)
    dec = np.abs(mx.dq_1x32(p, sc))[np.arange(500), i]
    e = sc[:, 0].astype(np.int64) - 127
    sat = dec == 448.0 * 2.0 ** e
    rel = np.abs(dec - amax) / amax
    assert np.all(sat | (rel <= 2.0 ** -4))
    # saturation happens exactly when amax * 2^-e rounds above 448
    assert np.array_equal(sat & (amax * 2.0 ** -e > 448), amax * 2.0 ** -e > 448)


def test_golden_block_example():
    """A hand-worked 32-element block (tests/golden/mx_block_example.txt)."""
    rows = np.loadtxt(os.path.join(GOLDEN, "mx_block_example.txt"),
                      comments="#")
    x = rows[:, 0]
    want_codes = rows[:, 1].astype(np.uint8)
    p, sc = mx.quantize_1x32(x[None, :])
    assert sc[0, 0] == 120          # amax 3.5 -> floor(log2) = 1 -> e = -7
    assert np.array_equal(p[0], want_codes)


# ----------------------------------------------------- block structure pins
def test_square_transpose_invariance(rng):
    """quant32x32(X^T) == quant32x32(X)^T bytewise, scales transposed."""
    x = rng.standard_normal((96, 128)) * np.exp(rng.uniform(-3, 3, (96, 128)))
    p, sc = mx.quantize_32x32(x)
    pt, sct = mx.quantize_32x32(x.T)
    assert np.array_equal(pt, p.T)
    assert np.array_equal(sct, sc.T)


def test_square_block_equals_flat_1024_block(rng):
    """A 32x32 block quantizes like one 1024-element block (same amax)."""
    x = rng.standard_normal((32, 32))
    p, sc = mx.quantize_32x32(x)
    amax = np.abs(x).max()
    e, code = mx.scale_exponent(np.array([amax]))
    assert sc[0, 0] == code[0]
    assert np.array_equal(p, mx.e4m3_encode(np.ldexp(x, -e[0])))


def test_1x32_blocks_are_independent(rng):
    x = rng.standard_normal((4, 128))
    x[:, 32:64] *= 1000.0
    p, sc = mx.quantize_1x32(x)
    for b in range(4):
        pb, scb = mx.quantize_1x32(x[:, 32 * b:32 * b + 32])
        assert np.array_equal(pb, p[:, 32 * b:32 * b + 32])
        assert np.array_equal(scb[:, 0], sc[:, b])


def test_rows_quantizer_ragged_tail(rng):
    x = rng.standard_normal((70, 3))
    p, sc = mx.quantize_along_rows(x)
    assert sc.shape == (3, 3)
    # the short last block (rows 64..69) uses its own amax
    e, code = mx.scale_exponent(np.abs(x[64:]).max(axis=0))
    assert np.array_equal(sc[2], code)
    assert np.array_equal(p[64:], mx.e4m3_encode(np.ldexp(x[64:], -e)))


def test_zero_block_and_decode_identity(rng):
    x = np.zeros((2, 32))
    p, sc = mx.quantize_1x32(x)
    assert np.all(p == 0) and np.all(sc == 0)
    # decode identity x_hat = 2^(E8M0 - 127) * v on random data
    y = rng.standard_normal((8, 64))
    p, sc = mx.quantize_1x32(y)
    dec = mx.e4m3_decode(p) * np.repeat(2.0 ** (sc.astype(np.int64) - 127), 32, 1)
    assert np.array_equal(dec, mx.dq_1x32(p, sc))


def test_mx_gemm_is_exact_dequantized_gemm(rng):
    """Products of decoded operands are exact in fp64: the MX GEMM equals an
    exact rational evaluation on a small case."""
    from fractions import Fraction
    a = rng.standard_normal((3, 64)); b = rng.standard_normal((2, 64))
    pa, sa = mx.quantize_1x32(a); pb, sb = mx.quantize_1x32(b)
    d = mx.mx_gemm(pa, sa, pb, sb)
    da = mx.dq_1x32(pa, sa); db = mx.dq_1x32(pb, sb)
    for i in range(3):
        for j in range(2):
            exact = sum(Fraction(float(x)) * Fraction(float(y))
                        for x, y in zip(da[i], db[j]))
            assert Fraction(float(d[i, j])) == exact


# ------------------------------------------------------------ layout pins
def test_mma_atom_is_a_permutation():
    r, kb = np.meshgrid(np.arange(128), np.arange(4), indexing="ij")
    off = layouts.atom_offset(r, kb).ravel()
    assert sorted(off.tolist()) == list(range(512))


def test_sf_row_starts_varlen():
    cu = np.array([0, 5, 133, 261, 262])
    assert layouts.sf_row_starts(cu).tolist() == [0, 128, 256, 384, 512]


# ----------------------------------------------------- quantizing GEMM epilogue
@pytest.mark.parametrize("block", ["1x32", "32x32"])
def test_gemm_quantize_layouts(block, rng):
    M, N = 256, 384
    d = rng.standard_normal((M, N)) * np.exp(rng.uniform(-3, 3, (M, 1)))
    out = layouts.gemm_quantize(d, block)
    # every tile byte is the compact code of its (row, block)
    sc_rows = out["sf"] if block == "1x32" else np.repeat(out["sf"], 32, axis=0)
    r, kb = np.meshgrid(np.arange(M), np.arange(N // 32), indexing="ij")
    assert np.array_equal(out["sf_mma"][r // 128, kb // 4, layouts.atom_offset(r % 128, kb % 4)],
                          sc_rows)
    if block == "32x32":
        # transpose invariance of square blocks: quantizing d^T gives the
        # transposed payload, and its row arrangement is sf_mma_t
        t = layouts.gemm_quantize(d.T, "32x32")
        assert np.array_equal(t["payload"], out["payload"].T)
        assert np.array_equal(t["sf_mma"], out["sf_mma_t"])


# ------------------------------------------------- other MX element formats
def _golden_formats():
    rows, e2m1 = {}, None
    with open(os.path.join(GOLDEN, "mx_element_formats.txt")) as fh:
        for line in fh:
            t = line.split()
            if not t or t[0].startswith("#"):
                continue
            if t[0] == "e2m1_values":
                e2m1 = [float(v) for v in t[1:]]
            else:
                rows[t[0]] = tuple(float(v) for v in t[1:])
    return rows, e2m1


def test_element_format_landmarks_match_golden():
    rows, e2m1 = _golden_formats()
    for fmt, (mx_max, mn_norm, mn_sub, emax, n) in rows.items():
        t = mx.fmt_table(fmt)
        fin = t[np.isfinite(t)]
        assert len(t) == n and fin.max() == mx_max and fin[fin > 0].min() == mn_sub
        eb, mb, bias, fe, _ = mx.FORMATS[fmt]
        assert fe == emax and _fmt_min_normal(fmt) == mn_norm
    assert list(mx.fmt_table("e2m1")[:8]) == e2m1


def _fmt_min_normal(fmt):
    eb, mb, bias, _, _ = mx.FORMATS[fmt]
    return mx.fmt_table(fmt)[1 << mb]          # exponent field 1, mantissa 0


def test_e5m2_decode_matches_torch_all_codes():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e5m2).to(torch.float64).numpy()
    ours = mx.fmt_table("e5m2")
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(ours[ok], ref[ok])


@pytest.mark.parametrize("fmt", ["e5m2", "e3m2", "e2m3", "e2m1"])
def test_element_encode_is_nearest_even_with_saturation(fmt, rng):
    t = mx.fmt_table(fmt)
    nbits = int(np.log2(len(t)))
    pos = t[:len(t) // 2]
    fin = np.isfinite(pos)
    vmax = pos[fin].max()
    x = np.concatenate([rng.standard_normal(3000) * vmax / 2, rng.uniform(-2 * vmax, 2 * vmax, 500),
                        (pos[fin][1:] + pos[fin][:-1]) / 2,       # exact midpoints
                        -(pos[fin][1:] + pos[fin][:-1]) / 2, [0.0, -0.0]])
    got = mx.fmt_encode(x, fmt)
    for xi, c in zip(x, got):
        a = min(abs(xi), vmax)
        d = np.abs(pos[fin] - a)
        best = np.flatnonzero(d == d.min())
        want = best[0] if len(best) == 1 else best[best % 2 == 0][0]
        assert (c & ((1 << (nbits - 1)) - 1)) == want
        assert bool(c >> (nbits - 1)) == bool(np.signbit(xi))


def test_e5m2_encode_matches_torch_in_range(rng):
    x = rng.standard_normal(4000) * np.exp(rng.uniform(-12, 12, 4000))
    x = x[np.abs(x) <= 57344.0]
    ref = torch.from_numpy(x).to(torch.float8_e5m2).view(torch.uint8).numpy()
    assert np.array_equal(mx.fmt_encode(x, "e5m2"), ref)


@pytest.mark.parametrize("fmt", ["e5m2", "e3m2", "e2m3", "e2m1"])
def test_scale_rule_per_format(fmt):
    emax = mx.FORMATS[fmt][3]
    for k in range(-40, 41, 7):
        e, code = mx.scale_exponent(np.array([1.5 * 2.0 ** k]), emax)
        assert e[0] == max(k - emax, -127) and code[0] == e[0] + 127
    # the block maximum lands in the top binade of the format: amax * 2^-e
    # in [2^emax, 2^(emax+1))
    x = np.random.default_rng(3).standard_normal((50, 32)) * 7.0
    p, sc = mx.quantize_1x32(x, fmt)
    amax = np.abs(x).max(axis=1)
    r = amax * 2.0 ** -(sc.astype(np.int64)[:, 0] - 127)
    assert np.all((r >= 2.0 ** emax) & (r < 2.0 ** (emax + 1)))


@pytest.mark.parametrize("a_fmt,b_fmt", [("e2m1", "e2m1"), ("e3m2", "e2m3"), ("e5m2", "e4m3")])
def test_mx_gemm_mixed_formats_exact(a_fmt, b_fmt):
    """The oracle GEMM of operands in other element formats against exact
    rational arithmetic on a small case (every decoded value is a dyadic
    rational, so the exact product sums are fractions)."""
    from fractions import Fraction
    rng = np.random.default_rng(11)
    a = rng.standard_normal((4, 64))
    b = rng.standard_normal((3, 64)) * 3.0
    pa, sa = mx.quantize_1x32(a, a_fmt)
    pb, sb = mx.quantize_1x32(b, b_fmt)
    got = mx.mx_gemm(pa, sa, pb, sb, a_fmt, b_fmt)
    ta, tb = mx.fmt_table(a_fmt), mx.fmt_table(b_fmt)
    for i in range(4):
        for j in range(3):
            acc = Fraction(0)
            for k in range(64):
                va = Fraction(ta[pa[i, k]]) * Fraction(2) ** (int(sa[i, k // 32]) - 127)
                vb = Fraction(tb[pb[j, k]]) * Fraction(2) ** (int(sb[j, k // 32]) - 127)
                acc += va * vb
            assert abs(Fraction(got[i, j]) - acc) <= abs(acc) * Fraction(1, 2 ** 50)


def test_mma_operand_bytes_hand_worked():
    """Packed FP4 / FP6 operand groups worked by hand from the bit-stream
    rule (code j at bits b*j.., little-endian, zero padding to 16 bytes)."""
    from oracle import layouts
    c4 = (np.arange(32) % 16).astype(np.uint8).reshape(1, 32)
    want4 = [0x10, 0x32, 0x54, 0x76, 0x98, 0xBA, 0xDC, 0xFE] + [0] * 8
    assert layouts.mma_operand_bytes(c4, "e2m1")[0, :16].tolist() == want4
    assert layouts.mma_operand_bytes(c4, "e2m1")[0, 16:].tolist() == want4
    # FP6: code 0x3F in slot 0 -> byte 0 = 0x3F; in slot 1 -> bits 6..11:
    # byte 0 = 0xC0, byte 1 = 0x0F; in slot 15 -> bits 90..95: byte 11 = 0xFC
    for slot, want in ((0, {0: 0x3F}), (1, {0: 0xC0, 1: 0x0F}), (15, {11: 0xFC})):
        c6 = np.zeros((1, 16), dtype=np.uint8)
        c6[0, slot] = 0x3F
        got = layouts.mma_operand_bytes(c6, "e3m2")[0]
        assert {i: int(v) for i, v in enumerate(got) if v} == want, slot
    # the sign bit of a code stays inside its own field
    c6 = np.zeros((1, 16), dtype=np.uint8)
    c6[0, 2] = 0x20                       # FP6 sign alone, slot 2 -> bit 17
    assert layouts.mma_operand_bytes(c6, "e2m3")[0, 2] == 0x02
    assert np.array_equal(layouts.mma_operand_bytes(c4, "e5m2"), c4)


def test_nvfp4_hand_worked_block():
    """One 16-element NVFP4 block by hand: amax = 3, s = E4M3(3/6 = 0.5) =
    0.5 (exact), elements x / 0.5 rounded to E2M1 {0, .5, 1, 1.5, 2, 3, 4, 6}
    with ties to the even code."""
    x = np.array([3.0, -3.0, 0.5, 0.25, 0.125, 1.1, 0.8, 0.0,
                  -0.375, 2.5, 1.75, 0.62, -1.0, 0.3, 0.9, 1.5])
    codes, sc = mx.quantize_nvfp4(x)
    assert sc.tolist() == [mx.e4m3_encode(0.5)]          # 0.5 = code 0x30
    y = x / 0.5
    # y: 6 -6 1 .5 .25 2.2 1.6 0 -.75 5 3.5 1.24 -2 .6 1.8 3
    want = [6.0, -6.0, 1.0, 0.5, 0.0, 2.0, 1.5, 0.0, -1.0, 4.0, 4.0, 1.0, -2.0, 0.5, 2.0, 3.0]
    got = mx.fmt_table("e2m1")[codes]
    assert got.tolist() == want
    # ties: 0.25 -> 0 (even code 0, not 0.5 = code 1); -0.75 -> -1 (code 2,
    # even, not -0.5 code 1); 5 -> 4 (code 6, even, not 6 = code 7); 3.5 -> 4
    assert np.array_equal(mx.dq_nvfp4(codes, sc), np.array(want) * 0.5)


def test_nvfp4_scale_rounding_and_zero_block():
    """amax = 6 * 0.3 = 1.8: s = E4M3(0.3) = 0.3125 (0.3 lies between 0.28125
    and 0.3125, nearer the latter), so the largest element 1.8 / 0.3125 =
    5.76 rounds to 6.  An all-zero block has scale code 0 and zero codes."""
    x = np.zeros((2, 16))
    x[0, 0] = 1.8
    codes, sc = mx.quantize_nvfp4(x)
    assert mx.e4m3_decode(sc[0]) == 0.3125
    assert mx.fmt_table("e2m1")[codes[0, 0]] == 6.0
    assert sc[1] == 0 and not codes[1].any()


def test_fp4_dense_bytes_hand_worked():
    from oracle import layouts
    c = np.array([[1, 2, 0xF, 0, 7, 8]], dtype=np.uint8)
    assert layouts.fp4_dense_bytes(c).tolist() == [[0x21, 0x0F, 0x87]]
