"""The inputs of the GPU test for the half-tile reference moves really reach
every route of the kernel's softmax (CPU only: a float64 restatement of the
kernel's control decisions, not of the method's arithmetic)."""
import math

import pytest

from online_softmax_tiling_gb300 import synth
from tests import parity


@pytest.mark.parametrize("dtype", [synth.FP16, synth.BF16])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_growing_halves_reach_every_route(dtype, d, causal):
    q, k, _ = parity.keys_growing_by_half(dtype, d)
    full, half2, common = parity.softmax_paths(q, k, dtype, 1.0 / math.sqrt(d), causal)
    # every row's first tile takes the full route; later tiles take all three
    assert full > 2000 + 300 and half2 > 500 and common > 3000, (full, half2, common)


def test_routes_of_plain_inputs_are_common():
    """iid N(0,1) inputs: after a row's first tile the reference never moves."""
    q = synth.tensor_bits(5, (1, 1, 512, 64), synth.BF16)
    k = synth.tensor_bits(6, (1, 1, 512, 64), synth.BF16)
    full, half2, common = parity.softmax_paths(q, k, synth.BF16, 0.125, False)
    assert (full, half2, common) == (512, 0, 3 * 512)
