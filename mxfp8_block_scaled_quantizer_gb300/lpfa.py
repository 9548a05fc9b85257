"""Thin ctypes binding of liblpfa.so (the C ABI in include/lpfa.h).

Argument marshalling only: every step of the attention path runs in the
library's CUDA kernels.  torch supplies device memory and the current
stream.  Importing this module fails loudly when liblpfa.so has not been
built; there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import math
import os
from dataclasses import dataclass
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liblpfa.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with "
        "`python -m mxfp8_block_scaled_quantizer_gb300._builder` (needs nvcc).")
_lib = ctypes.CDLL(LIB_PATH)

LPFA_OK, LPFA_ERR_INVALID_ARG, LPFA_ERR_UNSUPPORTED, LPFA_ERR_CUDA, \
    LPFA_ERR_TIMEOUT = range(5)
LPFA_BLK_1X32, LPFA_BLK_32X1, LPFA_BLK_32X32 = range(3)
LPFA_ELEM_E4M3, LPFA_ELEM_E5M2, LPFA_ELEM_E3M2, LPFA_ELEM_E2M3, LPFA_ELEM_E2M1 = range(5)
from . import FWD_KV_TILE  # noqa: E402  (key tile of the forward softmax)

_vp = ctypes.c_void_p
_i64 = ctypes.c_int64


class lpfa_seqs(ctypes.Structure):
    _fields_ = [("nseq", _i64), ("seqlen", _i64), ("total_tokens", _i64),
                ("total_sf_rows", _i64), ("cu_seqlens", _vp),
                ("cu_sf_rows", _vp)]


class lpfa_attn_desc(ctypes.Structure):
    _fields_ = [("seqs", lpfa_seqs), ("heads_q", _i64), ("heads_kv", _i64),
                ("head_dim", _i64), ("softmax_scale", ctypes.c_float),
                ("causal", ctypes.c_int32),
                ("rescale_threshold", ctypes.c_float),
                ("dq_static_scale", ctypes.c_float)]


def _sig(name, restype, *argtypes):
    f = getattr(_lib, name)
    f.restype = restype
    f.argtypes = list(argtypes)
    return f


_status_string = _sig("lpfa_status_string", ctypes.c_char_p, ctypes.c_int)
lpfa_version = _sig("lpfa_version", ctypes.c_int)
_device_supported = _sig("lpfa_device_supported", ctypes.c_int)
_varlen_sf_rows = _sig("lpfa_varlen_sf_rows", ctypes.c_int, _vp, _i64, _vp, _vp)
_mx_quantize = _sig("lpfa_mx_quantize", ctypes.c_int,
                    ctypes.POINTER(lpfa_seqs), _vp, _i64, _i64, ctypes.c_int,
                    _vp, _vp, _vp, _vp, _vp)
_mx_quantize_fmt = _sig("lpfa_mx_quantize_fmt", ctypes.c_int,
                        ctypes.POINTER(lpfa_seqs), _vp, _i64, _i64, ctypes.c_int, ctypes.c_int,
                        _vp, _vp, _vp, _vp, _vp)
_rms_quantize = _sig("lpfa_rmsnorm_mx_quantize", ctypes.c_int,
                     ctypes.POINTER(lpfa_seqs), _vp, _vp, _i64, _i64, ctypes.c_float,
                     ctypes.c_int, _vp, _vp, _vp, _vp, _vp, _vp)
class lpfa_gemm_problem(ctypes.Structure):
    _fields_ = [("a", _vp), ("sfa_mma", _vp), ("b", _vp), ("sfb_mma", _vp), ("d", _vp),
                ("M", _i64), ("N", _i64), ("K", _i64)]


_mx_gemm_grouped = _sig("lpfa_mx_gemm_grouped", ctypes.c_int, ctypes.POINTER(lpfa_gemm_problem),
                        ctypes.c_int32, _vp)
_mx_gemm = _sig("lpfa_mx_gemm", ctypes.c_int, _vp, _vp, _vp, _vp, _vp,
                _i64, _i64, _i64, _vp)
_mx_gemm_q = _sig("lpfa_mx_gemm_quantize", ctypes.c_int, _vp, _vp, _vp, _vp, _i64, _i64, _i64,
                  ctypes.c_int, _vp, _vp, _vp, _vp, _vp, _vp)
_mx_gemm_fmt = _sig("lpfa_mx_gemm_fmt", ctypes.c_int, _vp, _vp, _vp, _vp, _vp,
                    _i64, _i64, _i64, ctypes.c_int, ctypes.c_int, _vp)
_pack_operand = _sig("lpfa_mx_pack_operand", ctypes.c_int, _vp, _i64, _i64, ctypes.c_int,
                     _vp, _vp)
_gemm_fp4 = _sig("lpfa_mx_gemm_fp4", ctypes.c_int, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64,
                 ctypes.c_int, _vp)
_pack_fp4 = _sig("lpfa_fp4_pack_dense", ctypes.c_int, _vp, _i64, _i64, _vp, _vp)
_nvfp4_q = _sig("lpfa_nvfp4_quantize", ctypes.c_int, _vp, _i64, _i64, _vp, _vp, _vp, _vp)
_quant_t = _sig("lpfa_mx_quantize_t", ctypes.c_int, _vp, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _vp)
_norm_bwd_q = _sig("lpfa_rmsnorm_bwd_mx_quantize", ctypes.c_int, _vp, _vp, _vp, _vp, _i64, _i64,
                   _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp)
_mma_peak = _sig("lpfa_mma_peak", ctypes.c_int, ctypes.POINTER(ctypes.c_double), _vp)
_fwd_ws = _sig("lpfa_fwd_workspace_size", ctypes.c_size_t,
               ctypes.POINTER(lpfa_attn_desc))
_bwd_ws = _sig("lpfa_bwd_workspace_size", ctypes.c_size_t,
               ctypes.POINTER(lpfa_attn_desc))
_fwd = _sig("lpfa_fwd", ctypes.c_int, ctypes.POINTER(lpfa_attn_desc),
            _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp)
_bwd = _sig("lpfa_bwd", ctypes.c_int, ctypes.POINTER(lpfa_attn_desc),
            _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
            _vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp)
_fwd_bf16 = _sig("lpfa_fwd_bf16", ctypes.c_int, ctypes.POINTER(lpfa_attn_desc),
                 _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp)
_bwd_bf16 = _sig("lpfa_bwd_bf16", ctypes.c_int, ctypes.POINTER(lpfa_attn_desc),
                 _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp)
_fwd_expiry = _sig("lpfa_fwd_wait_expiry_selftest", ctypes.c_int,
                   ctypes.POINTER(lpfa_attn_desc), _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                   _vp, _vp, ctypes.c_size_t, ctypes.c_uint32, _vp)
_check = _sig("lpfa_check", ctypes.c_int, _vp, _vp)
_bwd_noalloc = _sig("lpfa_bwd_noalloc", ctypes.c_int,
                    ctypes.POINTER(lpfa_attn_desc), _vp, _vp, _vp, _vp, _vp,
                    _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                    _vp)

#: every symbol include/lpfa.h declares
EXPORTED = ("lpfa_status_string", "lpfa_version", "lpfa_device_supported",
            "lpfa_varlen_sf_rows", "lpfa_mx_quantize", "lpfa_mx_quantize_fmt",
            "lpfa_rmsnorm_mx_quantize",
            "lpfa_mx_gemm", "lpfa_mx_gemm_quantize",
            "lpfa_fwd_workspace_size", "lpfa_bwd_workspace_size", "lpfa_fwd",
            "lpfa_bwd", "lpfa_check", "lpfa_bwd_noalloc",
            "lpfa_fwd_wait_expiry_selftest", "lpfa_mma_peak", "lpfa_fwd_bf16",
            "lpfa_bwd_bf16", "lpfa_mx_gemm_fmt", "lpfa_mx_pack_operand",
            "lpfa_mx_gemm_fp4", "lpfa_fp4_pack_dense", "lpfa_nvfp4_quantize",
            "lpfa_mx_quantize_t", "lpfa_rmsnorm_bwd_mx_quantize", "lpfa_mx_gemm_grouped")


class LpfaError(RuntimeError):
    def __init__(self, status: int, call: str):
        self.status = status
        super().__init__(f"{call}: {lpfa_status_string(status)}")


def lpfa_status_string(status: int) -> str:
    return _status_string(status).decode()


def _ok(status: int, call: str):
    if status != LPFA_OK:
        raise LpfaError(status, call)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


# ---------------------------------------------------------------- sequences
@dataclass
class Seqs:
    """Sequence layout of token-major tensors (see lpfa_seqs)."""
    nseq: int
    seqlen: int
    total_tokens: int
    total_sf_rows: int
    cu_seqlens: Optional[torch.Tensor] = None   # device int32 [nseq+1]
    cu_sf_rows: Optional[torch.Tensor] = None   # device int32 [nseq+1]

    def c(self) -> lpfa_seqs:
        return lpfa_seqs(self.nseq, self.seqlen, self.total_tokens,
                         self.total_sf_rows, _ptr(self.cu_seqlens),
                         _ptr(self.cu_sf_rows))


def dense_seqs(batch: int, seqlen: int) -> Seqs:
    pad = -(-seqlen // 128) * 128
    return Seqs(batch, seqlen, batch * seqlen, batch * pad)


def varlen_seqs(cu_seqlens: torch.Tensor, lengths=None) -> Seqs:
    """cu_seqlens: int32 prefix offsets (device or host).  The padded scale
    row offsets are computed on the device by lpfa_varlen_sf_rows; the total
    padded row count comes from the host copy of the lengths."""
    cu_host = cu_seqlens.detach().to("cpu", torch.int64)
    lens = cu_host[1:] - cu_host[:-1]
    nseq = int(lens.numel())
    total_sf = int(((lens + 127) // 128 * 128).sum())
    cu_dev = cu_seqlens.to(device="cuda", dtype=torch.int32).contiguous()
    cu_sf = torch.empty(nseq + 1, dtype=torch.int32, device="cuda")
    lpfa_varlen_sf_rows(cu_dev, nseq, cu_sf)
    return Seqs(nseq, int(lens.max()), int(cu_host[-1]), total_sf, cu_dev,
                cu_sf)


def lpfa_varlen_sf_rows(cu_seqlens: torch.Tensor, nseq: int,
                        cu_sf_rows: torch.Tensor, stream=None):
    _ok(_varlen_sf_rows(_ptr(cu_seqlens), nseq, _ptr(cu_sf_rows),
                        _stream(stream)), "lpfa_varlen_sf_rows")


def lpfa_device_supported() -> bool:
    return _device_supported() == LPFA_OK


# ---------------------------------------------------------------- quantizer
@dataclass
class MXTensor:
    """E4M3 payload plus its E8M0 scales (compact and tensor-core layouts)."""
    data: torch.Tensor          # uint8 [T, H, D]
    sf: Optional[torch.Tensor]
    sf_mma: Optional[torch.Tensor]
    sf_mma_t: Optional[torch.Tensor]
    block: int
    seqs: Seqs


def lpfa_mx_quantize(seqs: Seqs, x: torch.Tensor, block: int,
                     out: torch.Tensor, sf=None, sf_mma=None, sf_mma_t=None,
                     stream=None, fmt: int = LPFA_ELEM_E4M3):
    """Raw call: x bf16 [T, H, D] (contiguous, CUDA); outputs preallocated;
    fmt selects the element format (E4M3 through lpfa_mx_quantize)."""
    assert x.is_cuda and x.dtype == torch.bfloat16 and x.is_contiguous()
    T, H, D = x.shape
    sc = seqs.c()
    if fmt == LPFA_ELEM_E4M3:
        _ok(_mx_quantize(ctypes.byref(sc), _ptr(x), H, D, block, _ptr(out),
                         _ptr(sf), _ptr(sf_mma), _ptr(sf_mma_t), _stream(stream)),
            "lpfa_mx_quantize")
    else:
        _ok(_mx_quantize_fmt(ctypes.byref(sc), _ptr(x), H, D, block, fmt, _ptr(out),
                             _ptr(sf), _ptr(sf_mma), _ptr(sf_mma_t), _stream(stream)),
            "lpfa_mx_quantize_fmt")


def mx_quantize(x: torch.Tensor, block: int, seqs: Optional[Seqs] = None,
                compact: bool = True, mma: bool = True,
                stream=None, fmt: int = LPFA_ELEM_E4M3) -> MXTensor:
    """Quantize bf16 [B, S, H, D] or packed [T, H, D] (``seqs`` for a jagged
    batch, else one sequence)."""
    if x.dim() == 4:
        B, S, H, D = x.shape
        if seqs is None:
            seqs = dense_seqs(B, S)
        x = x.reshape(B * S, H, D)
    T, H, D = x.shape
    if seqs is None:
        seqs = dense_seqs(1, T)
    x = x.contiguous()
    Tp = seqs.total_sf_rows
    dev = x.device
    out = torch.empty((T, H, D), dtype=torch.uint8, device=dev)
    sf = sf_mma = sf_mma_t = None
    if compact:
        shape = {LPFA_BLK_1X32: (T, H, D // 32), LPFA_BLK_32X1: (Tp // 32, H, D),
                 LPFA_BLK_32X32: (Tp // 32, H, D // 32)}[block]
        sf = torch.empty(shape, dtype=torch.uint8, device=dev)
    if mma:
        sf_mma = torch.empty((Tp // 128, H, 512), dtype=torch.uint8, device=dev)
        if block == LPFA_BLK_32X32:
            sf_mma_t = torch.empty((Tp // 128, H, 512), dtype=torch.uint8,
                                   device=dev)
    lpfa_mx_quantize(seqs, x, block, out, sf, sf_mma, sf_mma_t, stream, fmt)
    return MXTensor(out, sf, sf_mma, sf_mma_t, block, seqs)


def lpfa_rmsnorm_mx_quantize(seqs: Seqs, x: torch.Tensor, weight: torch.Tensor, eps: float,
                             block: int, out: torch.Tensor, sf=None, sf_mma=None,
                             sf_mma_t=None, rstd=None, stream=None):
    """Raw call: x bf16 [T, H, D], weight bf16 [H * D] (contiguous, CUDA);
    outputs preallocated."""
    assert x.is_cuda and x.dtype == torch.bfloat16 and x.is_contiguous()
    assert weight.dtype == torch.bfloat16 and weight.is_contiguous()
    T, H, D = x.shape
    assert weight.numel() == H * D
    sc = seqs.c()
    _ok(_rms_quantize(ctypes.byref(sc), _ptr(x), _ptr(weight), H, D, float(eps), block,
                      _ptr(out), _ptr(sf), _ptr(sf_mma), _ptr(sf_mma_t), _ptr(rstd),
                      _stream(stream)), "lpfa_rmsnorm_mx_quantize")


def rmsnorm_mx_quantize(x: torch.Tensor, weight: torch.Tensor, eps: float, block: int,
                        seqs: Optional[Seqs] = None, compact: bool = True,
                        mma: bool = True, stream=None):
    """Fused RMSNorm + MX quantization of bf16 [B, S, H, D] or packed
    [T, H, D] (``seqs`` for a jagged batch, else one sequence); the norm runs
    over each token's H * D values.  Returns (MXTensor of y, rstd fp32 [T])."""
    if x.dim() == 4:
        B, S, H, D = x.shape
        if seqs is None:
            seqs = dense_seqs(B, S)
        x = x.reshape(B * S, H, D)
    T, H, D = x.shape
    if seqs is None:
        seqs = dense_seqs(1, T)
    x = x.contiguous()
    Tp = seqs.total_sf_rows
    dev = x.device
    out = torch.empty((T, H, D), dtype=torch.uint8, device=dev)
    sf = sf_mma = sf_mma_t = None
    if compact:
        shape = {LPFA_BLK_1X32: (T, H, D // 32), LPFA_BLK_32X32: (Tp // 32, H, D // 32)}[block]
        sf = torch.empty(shape, dtype=torch.uint8, device=dev)
    if mma:
        sf_mma = torch.empty((Tp // 128, H, 512), dtype=torch.uint8, device=dev)
        if block == LPFA_BLK_32X32:
            sf_mma_t = torch.empty((Tp // 128, H, 512), dtype=torch.uint8, device=dev)
    rstd = torch.empty((T,), dtype=torch.float32, device=dev)
    lpfa_rmsnorm_mx_quantize(seqs, x, weight.contiguous(), eps, block, out, sf, sf_mma,
                             sf_mma_t, rstd, stream)
    return MXTensor(out, sf, sf_mma, sf_mma_t, block, seqs), rstd


# ---------------------------------------------------------------- GEMM
def lpfa_mx_gemm(a8, sfa_mma, b8, sfb_mma, d, stream=None):
    M, K = a8.shape
    N = b8.shape[0]
    _ok(_mx_gemm(_ptr(a8), _ptr(sfa_mma), _ptr(b8), _ptr(sfb_mma), _ptr(d),
                 M, N, K, _stream(stream)), "lpfa_mx_gemm")


def lpfa_mx_gemm_fmt(a, sfa_mma, b, sfb_mma, d, a_fmt, b_fmt, stream=None):
    """D = A B^T with A, B in the element formats a_fmt, b_fmt (LPFA_ELEM_*),
    operand bytes in the tensor core's layout ([M, K] / [N, K] bytes)."""
    M, K = a.shape
    N = b.shape[0]
    _ok(_mx_gemm_fmt(_ptr(a), _ptr(sfa_mma), _ptr(b), _ptr(sfb_mma), _ptr(d),
                     M, N, K, int(a_fmt), int(b_fmt), _stream(stream)), "lpfa_mx_gemm_fmt")


def mx_pack_operand(codes: torch.Tensor, fmt: int, out=None, stream=None) -> torch.Tensor:
    """One-code-per-byte [rows, cols] payload -> lpfa_mx_gemm_fmt operand bytes."""
    rows, cols = codes.shape
    if out is None:
        out = torch.empty_like(codes)
    _ok(_pack_operand(_ptr(codes), rows, cols, int(fmt), _ptr(out), _stream(stream)),
        "lpfa_mx_pack_operand")
    return out


def lpfa_mx_gemm_fp4(a, sfa_mma, b, sfb_mma, d, nvfp4: bool, stream=None):
    """D = A B^T on dense FP4 operands a [M, K/2], b [N, K/2] (kind::mxf4nvf4);
    MXFP4 (32-element E8M0 scales) or NVFP4 (16-element E4M3 scales)."""
    M, K2 = a.shape
    N = b.shape[0]
    _ok(_gemm_fp4(_ptr(a), _ptr(sfa_mma), _ptr(b), _ptr(sfb_mma), _ptr(d), M, N, 2 * K2,
                  int(bool(nvfp4)), _stream(stream)), "lpfa_mx_gemm_fp4")


def fp4_pack_dense(codes: torch.Tensor, stream=None) -> torch.Tensor:
    """One E2M1 code per byte [rows, cols] -> dense [rows, cols/2]."""
    rows, cols = codes.shape
    out = torch.empty((rows, cols // 2), dtype=torch.uint8, device=codes.device)
    _ok(_pack_fp4(_ptr(codes), rows, cols, _ptr(out), _stream(stream)), "lpfa_fp4_pack_dense")
    return out


def nvfp4_quantize(x: torch.Tensor, stream=None):
    """bf16 [rows, cols] -> (dense E2M1 [rows, cols/2], E4M3 scales
    [rows, cols/16], tensor-core scale tiles [rows/128, cols/64, 512] or None)."""
    assert x.is_cuda and x.dtype == torch.bfloat16 and x.is_contiguous()
    rows, cols = x.shape
    out = torch.empty((rows, cols // 2), dtype=torch.uint8, device=x.device)
    sf = torch.empty((rows, cols // 16), dtype=torch.uint8, device=x.device)
    mma = None
    if rows % 128 == 0 and cols % 64 == 0:
        mma = torch.empty((rows // 128, cols // 64, 512), dtype=torch.uint8, device=x.device)
    _ok(_nvfp4_q(_ptr(x), rows, cols, _ptr(out), _ptr(sf), _ptr(mma), _stream(stream)),
        "lpfa_nvfp4_quantize")
    return out, sf, mma


@dataclass
class MXT:
    """32x32 quantization with the payload in both orientations."""
    data: torch.Tensor      # [rows, cols]
    data_t: torch.Tensor    # [cols, rows_p]
    sf: torch.Tensor        # [rows_p/32, cols/32]
    sf_mma: torch.Tensor    # rows = rows: [rows_p/128, cols/128, 512]
    sf_mma_t: torch.Tensor  # rows = cols: [cols/128, rows_p/128, 512]


def _mxt_empty(rows, cols, dev) -> MXT:
    rp = -(-rows // 128) * 128
    u8 = dict(dtype=torch.uint8, device=dev)
    return MXT(torch.empty((rows, cols), **u8), torch.empty((cols, rp), **u8),
               torch.empty((rp // 32, cols // 32), **u8),
               torch.empty((rp // 128, cols // 128, 512), **u8),
               torch.empty((cols // 128, rp // 128, 512), **u8))


def mx_quantize_t(x: torch.Tensor, stream=None) -> MXT:
    """32x32 MX quantization of bf16 [rows, cols], payload in both orientations."""
    assert x.is_cuda and x.dtype == torch.bfloat16 and x.is_contiguous()
    rows, cols = x.shape
    m = _mxt_empty(rows, cols, x.device)
    _ok(_quant_t(_ptr(x), rows, cols, _ptr(m.data), _ptr(m.data_t), _ptr(m.sf), _ptr(m.sf_mma),
                 _ptr(m.sf_mma_t), _stream(stream)), "lpfa_mx_quantize_t")
    return m


def rmsnorm_bwd_mx_quantize(y, dz, gamma, rstd, stream=None):
    """dY of Z = RMSNorm(Y) gamma, 32x32-quantized in both orientations, and
    dgamma (fp32)."""
    rows, cols = y.shape
    m = _mxt_empty(rows, cols, y.device)
    rp = m.data_t.shape[1]
    part = torch.empty((rp // 32) * cols + rp, dtype=torch.float32, device=y.device)
    dgamma = torch.empty(cols, dtype=torch.float32, device=y.device)
    _ok(_norm_bwd_q(_ptr(y), _ptr(dz), _ptr(gamma), _ptr(rstd), rows, cols, _ptr(m.data),
                    _ptr(m.data_t), _ptr(m.sf), _ptr(m.sf_mma), _ptr(m.sf_mma_t), _ptr(part),
                    _ptr(dgamma), _stream(stream)), "lpfa_rmsnorm_bwd_mx_quantize")
    return m, dgamma


def gemm_norm_backward(xq: MXT, wq: MXT, y, rstd, gamma, dz, stream=None):
    """The jagged GEMM-Norm backward on MXFP8: xq = mx_quantize_t(X [T, K]),
    wq = mx_quantize_t(W [N, K]) (both may be kept from the forward), y the
    forward's bf16 Y [T, N], rstd fp32 [T], gamma bf16 [N], dz bf16 [T, N].
    Returns (dX fp32 [T, K], dW fp32 [N, K], dgamma fp32 [N])."""
    T, N = y.shape
    K = xq.data.shape[1]
    dyq, dgamma = rmsnorm_bwd_mx_quantize(y, dz, gamma, rstd, stream)
    dx = torch.empty((T, K), dtype=torch.float32, device=y.device)
    dw = torch.empty((N, K), dtype=torch.float32, device=y.device)
    lpfa_mx_gemm_grouped([(dyq.data, dyq.sf_mma, wq.data_t, wq.sf_mma_t, dx),
                          (dyq.data_t, dyq.sf_mma_t, xq.data_t, xq.sf_mma_t, dw)], stream)
    return dx, dw, dgamma


def lpfa_mx_gemm_grouped(problems, stream=None):
    """One or two D = A B^T MXFP8 GEMMs (fp32 out) in one launch; each
    problem is (a8 [M, K], sfa_mma, b8 [N, K], sfb_mma, d [M, N])."""
    arr = (lpfa_gemm_problem * len(problems))()
    for i, (a8, sfa, b8, sfb, d) in enumerate(problems):
        M, K = a8.shape
        arr[i] = lpfa_gemm_problem(_ptr(a8), _ptr(sfa), _ptr(b8), _ptr(sfb), _ptr(d),
                                   M, b8.shape[0], K)
    _ok(_mx_gemm_grouped(arr, len(problems), _stream(stream)), "lpfa_mx_gemm_grouped")


def lpfa_mx_gemm_quantize(a8, sfa_mma, b8, sfb_mma, block, out, sf=None, sf_mma=None,
                          sf_mma_t=None, d=None, stream=None):
    """Raw call: D = A B^T quantized in the epilogue; outputs preallocated."""
    M, K = a8.shape
    N = b8.shape[0]
    _ok(_mx_gemm_q(_ptr(a8), _ptr(sfa_mma), _ptr(b8), _ptr(sfb_mma), M, N, K, block,
                   _ptr(out), _ptr(sf), _ptr(sf_mma), _ptr(sf_mma_t), _ptr(d),
                   _stream(stream)), "lpfa_mx_gemm_quantize")


def mx_gemm_quantize(a8, sfa_mma, b8, sfb_mma, block: int, with_fp32: bool = False,
                     stream=None):
    """D = A B^T (block-scaled MXFP8 operands, 1x32 along K) quantized to
    MXFP8 in the epilogue.  Returns (payload [M, N], sf, sf_mma, sf_mma_t,
    d fp32 or None)."""
    M, K = a8.shape
    N = b8.shape[0]
    dev = a8.device
    out = torch.empty((M, N), dtype=torch.uint8, device=dev)
    shape = (M, N // 32) if block == LPFA_BLK_1X32 else (M // 32, N // 32)
    sf = torch.empty(shape, dtype=torch.uint8, device=dev)
    sf_mma = torch.empty((M // 128, N // 128, 512), dtype=torch.uint8, device=dev)
    sf_mma_t = (torch.empty((N // 128, M // 128, 512), dtype=torch.uint8, device=dev)
                if block == LPFA_BLK_32X32 else None)
    d = torch.empty((M, N), dtype=torch.float32, device=dev) if with_fp32 else None
    lpfa_mx_gemm_quantize(a8, sfa_mma, b8, sfb_mma, block, out, sf, sf_mma, sf_mma_t, d, stream)
    return out, sf, sf_mma, sf_mma_t, d


# ---------------------------------------------------------------- attention
def attn_desc(seqs: Seqs, heads_q: int, heads_kv: int, head_dim: int,
              causal: bool, softmax_scale: Optional[float] = None,
              rescale_threshold: float = 8.0,
              dq_static_scale: float = 1.0) -> lpfa_attn_desc:
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(head_dim)
    return lpfa_attn_desc(seqs.c(), heads_q, heads_kv, head_dim,
                          softmax_scale, int(bool(causal)), rescale_threshold,
                          dq_static_scale)


def fwd_workspace_size(desc: lpfa_attn_desc) -> int:
    return int(_fwd_ws(ctypes.byref(desc)))


def bwd_workspace_size(desc: lpfa_attn_desc) -> int:
    return int(_bwd_ws(ctypes.byref(desc)))


def lpfa_fwd(desc, q8, sfq, k8, sfk, v8, sfv, o, lse, ws, stream=None):
    _ok(_fwd(ctypes.byref(desc), _ptr(q8), _ptr(sfq), _ptr(k8), _ptr(sfk),
             _ptr(v8), _ptr(sfv), _ptr(o), _ptr(lse), _ptr(ws), ws.numel(),
             _stream(stream)), "lpfa_fwd")


def lpfa_bwd(desc, q8, sfq, sfq_t, k8, sfk, sfk_t, v8, sfv, do8, sfdo,
             sfdo_t, o, dout, lse, dq, dk, dv, ws, stream=None):
    _ok(_bwd(ctypes.byref(desc), _ptr(q8), _ptr(sfq), _ptr(sfq_t), _ptr(k8),
             _ptr(sfk), _ptr(sfk_t), _ptr(v8), _ptr(sfv), _ptr(do8),
             _ptr(sfdo), _ptr(sfdo_t), _ptr(o), _ptr(dout), _ptr(lse),
             _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws), ws.numel(),
             _stream(stream)), "lpfa_bwd")


def lpfa_fwd_bf16(desc, q, k, v, o, lse, ws, stream=None):
    _ok(_fwd_bf16(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                  _ptr(ws), ws.numel(), _stream(stream)), "lpfa_fwd_bf16")


def lpfa_bwd_bf16(desc, q, k, v, o, dout, lse, dq, dk, dv, ws, stream=None):
    _ok(_bwd_bf16(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout),
                  _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(ws), ws.numel(),
                  _stream(stream)), "lpfa_bwd_bf16")


def lpfa_fwd_wait_expiry_selftest(desc, q8, sfq, k8, sfk, v8, sfv, o, lse, ws,
                                  wait_limit_us, stream=None):
    _ok(_fwd_expiry(ctypes.byref(desc), _ptr(q8), _ptr(sfq), _ptr(k8), _ptr(sfk),
                    _ptr(v8), _ptr(sfv), _ptr(o), _ptr(lse), _ptr(ws), ws.numel(),
                    wait_limit_us, _stream(stream)), "lpfa_fwd_wait_expiry_selftest")


def lpfa_mma_peak(stream=None) -> float:
    """Block-scaled MXFP8 MMA rate of the tensor pipe (FLOP/s); synchronises."""
    v = ctypes.c_double(0.0)
    _ok(_mma_peak(ctypes.byref(v), _stream(stream)), "lpfa_mma_peak")
    return v.value


def lpfa_check(ws: torch.Tensor, stream=None):
    _ok(_check(_ptr(ws), _stream(stream)), "lpfa_check")


def check_status(ws: torch.Tensor, stream=None) -> int:
    """lpfa_check's status code, without raising."""
    return int(_check(_ptr(ws), _stream(stream)))


# ------------------------------------------------------- convenience layer
def _seqs_for(qt: torch.Tensor, B, S, cu_seqlens) -> "Seqs":
    """BSHD -> B dense sequences; packed [T, H, D] -> the cu_seqlens
    sequences, or one sequence of T tokens without them."""
    if cu_seqlens is not None:
        return varlen_seqs(cu_seqlens)
    if B is None:
        return dense_seqs(1, qt.shape[0])
    return dense_seqs(B, S)


def _as_tokens(x: torch.Tensor):
    """[B, S, H, D] -> ([B*S, H, D], B, S); [T, H, D] -> (x, None, None)."""
    if x.dim() == 4:
        B, S = x.shape[:2]
        return x.reshape(B * S, *x.shape[2:]).contiguous(), B, S
    return x.contiguous(), None, None


def quantize_forward_operands(q, k, v, seqs: Seqs, stream=None):
    """MX-quantize Q, K (1x32 along head_dim) and V (32 along tokens)."""
    mq = mx_quantize(q, LPFA_BLK_1X32, seqs, compact=False, stream=stream)
    mk = mx_quantize(k, LPFA_BLK_1X32, seqs, compact=False, stream=stream)
    mv = mx_quantize(v, LPFA_BLK_32X1, seqs, compact=False, stream=stream)
    return mq, mk, mv


def attention_forward_mx(mq: MXTensor, mk: MXTensor, mv: MXTensor,
                         desc: lpfa_attn_desc, out=None, lse=None, ws=None,
                         stream=None):
    """lpfa_fwd on already-quantized operands.  Returns (o, lse, ws)."""
    T, Hq, D = mq.data.shape
    dev = mq.data.device
    if out is None:
        out = torch.empty((T, Hq, D), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((Hq, T), dtype=torch.float32, device=dev)
    if ws is None:
        ws = torch.empty(fwd_workspace_size(desc), dtype=torch.uint8, device=dev)
    lpfa_fwd(desc, mq.data, mq.sf_mma, mk.data, mk.sf_mma, mv.data, mv.sf_mma,
             out, lse, ws, stream)
    return out, lse, ws


def mx_attention_forward(q, k, v, *, causal: bool, softmax_scale=None,
                         cu_seqlens: Optional[torch.Tensor] = None,
                         rescale_threshold: float = 8.0, check: bool = True):
    """Quantize and run the MXFP8 forward.  q [B,S,Hq,D] (or packed [T,Hq,D]
    with ``cu_seqlens``), k/v with Hkv heads, all bf16 CUDA tensors.
    Returns (o shaped like q, lse [Hq, T])."""
    shape = q.shape
    qt, B, S = _as_tokens(q)
    kt, _, _ = _as_tokens(k)
    vt, _, _ = _as_tokens(v)
    seqs = _seqs_for(qt, B, S, cu_seqlens)
    T, Hq, D = qt.shape
    desc = attn_desc(seqs, Hq, kt.shape[1], D, causal, softmax_scale,
                     rescale_threshold)
    mq, mk, mv = quantize_forward_operands(qt, kt, vt, seqs)
    o, lse, ws = attention_forward_mx(mq, mk, mv, desc)
    if check:
        lpfa_check(ws)
    return o.reshape(shape), lse


def attention_forward_bf16(q, k, v, desc: lpfa_attn_desc, out=None, lse=None, ws=None,
                           stream=None):
    """lpfa_fwd_bf16 on bf16 [T, H, D] operands.  Returns (o, lse, ws)."""
    T, Hq, D = q.shape
    dev = q.device
    if out is None:
        out = torch.empty((T, Hq, D), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((Hq, T), dtype=torch.float32, device=dev)
    if ws is None:
        ws = torch.empty(fwd_workspace_size(desc), dtype=torch.uint8, device=dev)
    lpfa_fwd_bf16(desc, q, k, v, out, lse, ws, stream)
    return out, lse, ws


def bf16_attention_forward(q, k, v, *, causal: bool, softmax_scale=None,
                           cu_seqlens: Optional[torch.Tensor] = None,
                           rescale_threshold: float = 8.0, check: bool = True):
    """The bf16 variant of mx_attention_forward (same kernel with kind::f16
    MMAs on bf16 operands, P rounded to bf16).  Returns (o, lse)."""
    shape = q.shape
    qt, B, S = _as_tokens(q)
    kt, _, _ = _as_tokens(k)
    vt, _, _ = _as_tokens(v)
    seqs = _seqs_for(qt, B, S, cu_seqlens)
    T, Hq, D = qt.shape
    desc = attn_desc(seqs, Hq, kt.shape[1], D, causal, softmax_scale,
                     rescale_threshold)
    o, lse, ws = attention_forward_bf16(qt, kt, vt, desc)
    if check:
        lpfa_check(ws)
    return o.reshape(shape), lse


def attention_backward_bf16(q, k, v, o, dout, lse, desc: lpfa_attn_desc, dq=None, dk=None,
                            dv=None, ws=None, stream=None):
    """lpfa_bwd_bf16 on bf16 [T, H, D] operands.  Returns (dq fp16, dk, dv, ws)."""
    T, Hq, D = q.shape
    Hkv = k.shape[1]
    dev = q.device
    if dq is None:
        dq = torch.empty((T, Hq, D), dtype=torch.float16, device=dev)
    if dk is None:
        dk = torch.empty((T, Hkv, D), dtype=torch.bfloat16, device=dev)
    if dv is None:
        dv = torch.empty((T, Hkv, D), dtype=torch.bfloat16, device=dev)
    if ws is None:
        ws = torch.empty(bwd_workspace_size(desc), dtype=torch.uint8, device=dev)
    lpfa_bwd_bf16(desc, q, k, v, o, dout, lse, dq, dk, dv, ws, stream)
    return dq, dk, dv, ws


def bf16_attention_backward(q, k, v, o, do, lse, *, causal: bool, softmax_scale=None,
                            cu_seqlens: Optional[torch.Tensor] = None,
                            dq_static_scale: float = 1.0, check: bool = True):
    """The bf16 variant of mx_attention_backward (head_dim 128).  Returns
    (dq fp16, dk, dv) shaped like q, k, v."""
    qt, B, S = _as_tokens(q)
    kt, _, _ = _as_tokens(k)
    vt, _, _ = _as_tokens(v)
    ot, _, _ = _as_tokens(o)
    dot, _, _ = _as_tokens(do)
    seqs = _seqs_for(qt, B, S, cu_seqlens)
    T, Hq, D = qt.shape
    desc = attn_desc(seqs, Hq, kt.shape[1], D, causal, softmax_scale,
                     dq_static_scale=dq_static_scale)
    dq, dk, dv, ws = attention_backward_bf16(qt, kt, vt, ot, dot, lse, desc)
    if check:
        lpfa_check(ws)
    return dq.reshape(q.shape), dk.reshape(k.shape), dv.reshape(v.shape)


def quantize_backward_operands(q, k, v, do, seqs: Seqs, stream=None):
    """MX-quantize Q, K, dO in square 32x32 blocks (both scale layouts) and V
    in 1x32 blocks along head_dim."""
    mq = mx_quantize(q, LPFA_BLK_32X32, seqs, compact=False, stream=stream)
    mk = mx_quantize(k, LPFA_BLK_32X32, seqs, compact=False, stream=stream)
    mdo = mx_quantize(do, LPFA_BLK_32X32, seqs, compact=False, stream=stream)
    mv = mx_quantize(v, LPFA_BLK_1X32, seqs, compact=False, stream=stream)
    return mq, mk, mv, mdo


def attention_backward_mx(mq: MXTensor, mk: MXTensor, mv: MXTensor,
                          mdo: MXTensor, o: torch.Tensor, dout: torch.Tensor,
                          lse: torch.Tensor, desc: lpfa_attn_desc, dq=None,
                          dk=None, dv=None, ws=None, stream=None):
    """lpfa_bwd on already-quantized operands.  o, dout: bf16 [T, Hq, D];
    lse: fp32 [Hq, T].  Returns (dq fp16, dk bf16, dv bf16, ws)."""
    T, Hq, D = mq.data.shape
    Hkv = mk.data.shape[1]
    dev = mq.data.device
    if dq is None:
        dq = torch.empty((T, Hq, D), dtype=torch.float16, device=dev)
    if dk is None:
        dk = torch.empty((T, Hkv, D), dtype=torch.bfloat16, device=dev)
    if dv is None:
        dv = torch.empty((T, Hkv, D), dtype=torch.bfloat16, device=dev)
    if ws is None:
        ws = torch.empty(bwd_workspace_size(desc), dtype=torch.uint8, device=dev)
    lpfa_bwd(desc, mq.data, mq.sf_mma, mq.sf_mma_t, mk.data, mk.sf_mma,
             mk.sf_mma_t, mv.data, mv.sf_mma, mdo.data, mdo.sf_mma,
             mdo.sf_mma_t, o.contiguous(), dout.contiguous(), lse.contiguous(),
             dq, dk, dv, ws, stream)
    return dq, dk, dv, ws


def mx_attention_backward(q, k, v, o, dout, lse, *, causal: bool,
                          softmax_scale=None,
                          cu_seqlens: Optional[torch.Tensor] = None,
                          dq_static_scale: float = 1.0, check: bool = True):
    """Quantize and run the MXFP8 backward.  Shapes as mx_attention_forward;
    o/dout like q, lse [Hq, T].  Returns (dq fp16, dk, dv) shaped like q/k/v."""
    shape_q, shape_k = q.shape, k.shape
    qt, B, S = _as_tokens(q)
    kt, _, _ = _as_tokens(k)
    vt, _, _ = _as_tokens(v)
    ot, _, _ = _as_tokens(o)
    dot, _, _ = _as_tokens(dout)
    seqs = _seqs_for(qt, B, S, cu_seqlens)
    T, Hq, D = qt.shape
    desc = attn_desc(seqs, Hq, kt.shape[1], D, causal, softmax_scale,
                     dq_static_scale=dq_static_scale)
    mq, mk, mv, mdo = quantize_backward_operands(qt, kt, vt, dot, seqs)
    dq, dk, dv, ws = attention_backward_mx(mq, mk, mv, mdo, ot, dot, lse, desc)
    if check:
        lpfa_check(ws)
    return dq.reshape(shape_q), dk.reshape(shape_k), dv.reshape(shape_k)


def lpfa_bwd_noalloc(desc, q8, sfq, sfq_t, k8, sfk, sfk_t, v8, sfv, do8, sfdo,
                     sfdo_t, o, dout, lse, dq, dk, dv, stream=None):
    """lpfa_bwd without a workspace argument: the library's static device
    scratch array stands in for it (for callers that cannot allocate)."""
    _ok(_bwd_noalloc(ctypes.byref(desc), _ptr(q8), _ptr(sfq), _ptr(sfq_t),
                     _ptr(k8), _ptr(sfk), _ptr(sfk_t), _ptr(v8), _ptr(sfv),
                     _ptr(do8), _ptr(sfdo), _ptr(sfdo_t), _ptr(o), _ptr(dout),
                     _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv), _stream(stream)),
        "lpfa_bwd_noalloc")
