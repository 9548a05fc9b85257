"""The C-ABI library builds, loads without a GPU, and exports every symbol
include/lpfa.h declares; host-side argument checks (no kernel launches)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lpfa.h")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(lpfa_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    from mxfp8_block_scaled_quantizer_gb300 import build
    build()
    from mxfp8_block_scaled_quantizer_gb300 import lpfa
    return lpfa


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("lpfa_mx_quantize", "lpfa_fwd", "lpfa_bwd", "lpfa_mx_gemm",
              "lpfa_check", "lpfa_varlen_sf_rows"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    so = ctypes.CDLL(lib.LIB_PATH)
    for name in _declared():
        assert hasattr(so, name), name
    assert set(lib.EXPORTED) == set(_declared())


def test_status_strings_and_version(lib):
    assert lib.lpfa_version() == 1
    assert lib.lpfa_status_string(0) == "LPFA_OK"
    assert lib.lpfa_status_string(4) == "LPFA_ERR_TIMEOUT"
    assert lib.lpfa_status_string(99) == "LPFA_ERR_UNKNOWN"


def test_invalid_arguments_rejected_before_launch(lib):
    """Null / misaligned pointers and bad shapes return INVALID_ARG on the
    host; nothing reaches the GPU (this runs without one)."""
    s = lib.lpfa_seqs(1, 128, 128, 128, None, None)
    st = lib._mx_quantize(ctypes.byref(s), None, 1, 128, 0, None, None, None,
                          None, None)
    assert st == lib.LPFA_ERR_INVALID_ARG
    bad = lib.lpfa_seqs(1, 128, 100, 128, None, None)   # T != nseq*seqlen
    st = lib._mx_quantize(ctypes.byref(bad), ctypes.c_void_p(16), 1, 128, 0,
                          ctypes.c_void_p(16), None, None, None, None)
    assert st == lib.LPFA_ERR_INVALID_ARG
    st = lib._mx_quantize(ctypes.byref(s), ctypes.c_void_p(18), 1, 128, 0,
                          ctypes.c_void_p(16), None, None, None, None)
    assert st == lib.LPFA_ERR_INVALID_ARG          # misaligned input
    st = lib._mx_quantize(ctypes.byref(s), ctypes.c_void_p(16), 1, 96, 0,
                          ctypes.c_void_p(16), None, None, None, None)
    assert st == lib.LPFA_ERR_UNSUPPORTED          # head_dim 96
    st = lib._mx_gemm(None, None, None, None, None, 128, 256, 128, None)
    assert st == lib.LPFA_ERR_INVALID_ARG


def test_new_entry_points_reject_bad_arguments_before_launch(lib):
    """The element-format quantizer, the fused RMSNorm quantizer and the
    quantizing GEMM check their arguments on the host (no GPU needed)."""
    s = lib.lpfa_seqs(1, 128, 128, 128, None, None)
    p = ctypes.c_void_p(256)                           # aligned, never dereferenced
    # element format outside the enum
    st = lib._mx_quantize_fmt(ctypes.byref(s), p, 1, 128, 0, 7, p, None, None, None, None)
    assert st == lib.LPFA_ERR_INVALID_ARG
    # transposed scale layout requested for 1x32 blocks
    st = lib._mx_quantize_fmt(ctypes.byref(s), p, 1, 128, 0, 1, p, None, None, p, None)
    assert st == lib.LPFA_ERR_INVALID_ARG
    # fused RMSNorm: eps <= 0, missing weight, 32x1 blocks, head_dim 96
    st = lib._rms_quantize(ctypes.byref(s), p, p, 1, 128, 0.0, 0, p, None, None, None, None, None)
    assert st == lib.LPFA_ERR_INVALID_ARG
    st = lib._rms_quantize(ctypes.byref(s), p, None, 1, 128, 1e-6, 0, p, None, None, None, None,
                           None)
    assert st == lib.LPFA_ERR_INVALID_ARG
    st = lib._rms_quantize(ctypes.byref(s), p, p, 1, 128, 1e-6, 1, p, None, None, None, None, None)
    assert st == lib.LPFA_ERR_UNSUPPORTED
    st = lib._rms_quantize(ctypes.byref(s), p, p, 1, 96, 1e-6, 0, p, None, None, None, None, None)
    assert st == lib.LPFA_ERR_UNSUPPORTED
    # quantizing GEMM: 32x1 blocks, shapes off the tile grid, null output
    st = lib._mx_gemm_q(p, p, p, p, 128, 256, 128, 1, p, None, None, None, None, None)
    assert st == lib.LPFA_ERR_UNSUPPORTED
    st = lib._mx_gemm_q(p, p, p, p, 128, 384, 128, 0, p, None, None, None, None, None)
    assert st == lib.LPFA_ERR_UNSUPPORTED          # N not a multiple of 256
    st = lib._mx_gemm_q(p, p, p, p, 128, 256, 128, 0, None, None, None, None, None, None)
    assert st == lib.LPFA_ERR_INVALID_ARG
    st = lib._mx_gemm_q(p, p, p, p, 128, 256, 128, 0, p, None, None, p, None, None)
    assert st == lib.LPFA_ERR_INVALID_ARG          # transposed layout with 1x32
