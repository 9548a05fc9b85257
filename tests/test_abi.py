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
