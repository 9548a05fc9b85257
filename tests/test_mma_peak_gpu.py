"""lpfa_mma_peak: the tensor pipe's block-scaled MXFP8 MMA rate.

The rate must be physically possible (below the tensor cores' issue limit,
8192 MACs per clock per SM at the highest SM clock) and not far below what
the GEMMs in the same process reach (a pipe-only measurement that came out
under a full GEMM would not be measuring the pipe)."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    from mxfp8_block_scaled_quantizer_gb300 import build
    build()
    from mxfp8_block_scaled_quantizer_gb300 import lpfa
    return lpfa


def test_mma_peak_is_physical(L):
    props = torch.cuda.get_device_properties(0)
    rate = L.lpfa_mma_peak()
    ceiling = 2.0 * 8192 * props.multi_processor_count * 2.2e9   # 2.2 GHz > max clock
    assert 1.0e15 < rate < ceiling, rate
    # the same again agrees within 10 % (a steady measurement)
    rate2 = L.lpfa_mma_peak()
    assert abs(rate2 - rate) < 0.1 * rate
