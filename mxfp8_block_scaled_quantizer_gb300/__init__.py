"""lpfa: MXFP8 block-scaled FlashAttention (forward and backward) for GB300.

The compute path is the CUDA library ``liblpfa.so`` (C ABI, include/lpfa.h);
this package holds its sources (``csrc/``), its build script (``_builder.py``)
and a thin ctypes binding (``lpfa.py``).  ``import
mxfp8_block_scaled_quantizer_gb300.lpfa`` raises if the library is missing.
"""
__all__ = ["build", "FWD_KV_TILE", "BWD_KV_TILE"]

# Keys per tile of the forward kernel's online softmax.  The running max, and
# with it the rounding of P to E4M3, moves once per tile, so a reference that
# wants the kernel's exact quantization points runs its online softmax over
# tiles of this size.
FWD_KV_TILE = 256

# Keys per CTA of the backward kernel; each CTA adds its FP16 dQ partial once
# per query step, so dQ is a sum of FP16-rounded partials over this many keys.
BWD_KV_TILE = 128


def build(verbose: bool = False, force: bool = False) -> str:
    from ._builder import build as _build
    return _build(verbose=verbose, force=force)
