"""CPU oracle for MXFP8 block-scaled attention (fp64, numpy).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline legs (``cpu_baseline`` and ``--impl reference``)
may import, call or execute anything in this package.  The product path (the
CUDA library and its Python binding) never imports it and shares no code,
tables or helpers with it; the only module both sides use is ``workloads``,
which draws the seeded inputs and holds none of the method's arithmetic.

Modules:
  mx         E4M3 / E8M0 codec and the 1x32, 32-along-tokens and 32x32 block
             quantizers.
  attention  exact fp64 attention (forward and gradients) and the
             quantization-matched MXFP8 forward / backward.
  layouts    the MMA-ready scale arrangements, written from the tensor-core
             scale-factor layout description, for checking the quantizer's
             second scale output.
  norm       RMSNorm followed by MX quantization (the fused producer).
  gemm_norm  the jagged GEMM-Norm backward (exact and at the MXFP8
             quantization points).
"""
from . import mx, attention, norm, gemm_norm  # noqa: F401
