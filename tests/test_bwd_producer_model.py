"""Host-side model of the backward producer's -log2 LSE / -D row ring.

The producer warp of ``mx_attn_bwd_kernel`` requests a step's rows
``kLseAhead`` steps before the step's Q / dO copies and builds the step's
accumulator seed from them ``kLag`` steps after those copies; the rows live in
``kLseSlots`` slots, each with its own mbarrier.  A slot may be refilled only
after the seed of its previous fill has been built (a refill before that would
arrive twice on the slot's mbarrier within one phase).  This test reads the
constants from the kernel source and replays the producer's program order.
"""
import os
import re

import pytest

SRC = os.path.join(os.path.dirname(__file__), "..", "mxfp8_block_scaled_quantizer_gb300", "csrc", "bwd.cu")


def _ring_constants(b16: bool):
    s = open(SRC).read()
    stages = re.search(r"kStages = B16 \? (\d+) : (\d+);", s)
    ahead = re.search(r"kLseAhead = kStages >= 4 \? (\d+) : (\d+);", s)
    lag = re.search(r"kLag = kStages >= 4 \? (\d+) : (\d+);", s)
    assert stages and ahead and lag, "ring constants not found in the kernel source"
    assert "kLseSlots = kLseAhead + kLag + 1;" in s
    n_stages = int(stages.group(1) if b16 else stages.group(2))
    deep = n_stages >= 4
    a = int(ahead.group(1) if deep else ahead.group(2))
    g = int(lag.group(1) if deep else lag.group(2))
    return a, g, a + g + 1


def replay(nsteps: int, ahead: int, lag: int, slots: int):
    """Producer order: rows of steps [0, ahead) first; then per iteration i the
    copies of step i, the rows of step i + ahead, the seed of step i - lag."""
    held = {}
    seeded = set()

    def fill(k):
        sl = k % slots
        if sl in held and held[sl] not in seeded:
            raise AssertionError(f"slot {sl} refilled with step {k} before the seed of step {held[sl]}")
        held[sl] = k

    def seed(j):
        if held.get(j % slots) != j:
            raise AssertionError(f"seed of step {j} reads the fill of step {held.get(j % slots)}")
        seeded.add(j)

    for j in range(min(ahead, nsteps)):
        fill(j)
    for i in range(nsteps + lag):
        if i + ahead < nsteps:
            fill(i + ahead)
        if i - lag >= 0:
            seed(i - lag)
    assert seeded == set(range(nsteps))


@pytest.mark.parametrize("b16", [False, True])
def test_lse_ring_never_refills_early(b16):
    a, g, slots = _ring_constants(b16)
    for n in range(0, 260):
        replay(n, a, g, slots)


def test_lse_ring_model_catches_a_short_ring():
    # three slots with rows two steps ahead and a one-step seed lag refill a
    # slot whose seed is still pending
    with pytest.raises(AssertionError, match="refilled"):
        replay(10, 2, 1, 3)
