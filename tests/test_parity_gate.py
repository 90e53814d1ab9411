"""The parity gates the GPU tests and the benchmark apply, checked on
planted errors (no GPU): the plain gate on the error beyond half an output
ulp, and the ceilinged gate kept for inputs widened on purpose."""
import numpy as np
import pytest

from online_softmax_tiling_gb300 import synth
from tests import parity


def _case(n=20000, err=None, spread=0.05, dtype=synth.BF16):
    rng = np.random.default_rng(3)
    o_ref = rng.uniform(0.25, 0.49, size=(n // 10, 10))      # half ulp (bf16) = 2^-10 here
    o = o_ref.copy()
    for idx, e in (err or {}).items():
        o.flat[idx] += e
    sp = np.full_like(o_ref, spread)
    lse = np.zeros(o_ref.shape[0])
    return parity.compare(synth.round_to_bits(o, dtype), lse.astype(np.float32), o_ref, lse, sp,
                          dtype)


def test_plain_gate_counts_only_output_rounding():
    st = _case()
    parity.assert_within(dict(st), "exact")
    hu = 2.0 ** -10
    st = _case(err={5: parity.MAX_EXCESS + 2 * hu})          # beyond half an ulp by > 4e-3
    assert st["n_excess_over_max"] == 1
    with pytest.raises(AssertionError):
        parity.assert_within(dict(st), "one element over")


def test_widened_gate_ceilings():
    # spread 1: the weight rounding may explain up to u/(1-u) = 3.9e-3 more
    over = parity.MAX_EXCESS + 2.5e-3
    st = _case(err={7: over}, spread=1.0)
    with pytest.raises(AssertionError):
        parity.assert_within(dict(st), "plain gate")
    parity.assert_within(dict(st), "widened", parity.WIDENED)
    # beyond both roundings: fails even the widened gate
    st = _case(err={7: parity.MAX_EXCESS + 6e-3}, spread=1.0)
    with pytest.raises(AssertionError):
        parity.assert_within(dict(st), "widened, too far", parity.WIDENED)
    # more than one element in ten thousand over 4e-3: fails the ceiling
    st = _case(err={i: over for i in range(0, 200, 20)}, spread=1.0)
    assert st["n_excess_over_max"] == 10 > parity.WIDENED.max_frac * st["n_elements"]
    with pytest.raises(AssertionError):
        parity.assert_within(dict(st), "widened, too many", parity.WIDENED)


def test_gate_for_workloads():
    assert parity.gate_for(synth.workload("C4")) is parity.WIDENED
    for name in ("C1", "C2", "C3", "C5", "C5r", "T_b2h32n4096d128_bf16", "T_b2h32n4096d128_fp16"):
        assert parity.gate_for(synth.workload(name)) is None
