"""bench.py's algorithmic counts (CPU only): FLOPs of the metric, 2^x
evaluations and L2 -> SM bytes per launch, pinned by closed forms and by the
bytes ncu measured for the fused and wide kernels."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
from online_softmax_tiling_gb300 import synth  # noqa: E402


def test_metric_flops_closed_form():
    """4 B H N^2 d, halved with the causal mask."""
    t = synth.workload("T_b2h32n4096d128_bf16")
    assert t.flops == 4 * 2 * 32 * 4096 ** 2 * 128
    c5 = synth.workload("C5")
    assert c5.flops == 4 * 1 * 8 * 16384 ** 2 * 128 // 2


def test_exp_count_is_one_per_visible_pair():
    t = bench.ceiling_counts(synth.workload("T_b2h32n4096d128_bf16"))
    assert t["exps"] == 2 * 32 * 4096 * 4096
    c3 = bench.ceiling_counts(synth.workload("C3"))
    assert c3["exps"] == 4 * 16 * 4096 * 4097 // 2


@pytest.mark.parametrize("name,measured,digits", [
    # l1tex__m_xbar2l1tex_read_bytes.sum of one launch as ncu printed it, in
    # GB with the printed number of decimals
    ("T_b2h32n4096d128_bf16", 2.214593, 6),
    ("D256", 4.362, 3),
])
def test_l2_bytes_match_the_measured_reads(name, measured, digits):
    """Each unit reads its Q tiles once and every K and V tile it visits."""
    got = bench.ceiling_counts(synth.workload(name))["l2_bytes"] / 1e9
    assert round(got, digits) == pytest.approx(measured), (got, measured)


def test_l2_bytes_closed_form_non_causal():
    """Two 128-row query tiles per unit for d <= 128: every unit reads all
    N / 128 key tiles of K and V, and each head's Q once."""
    B, H, N, d = 2, 32, 4096, 128
    units = B * H * (N // 256)
    want = units * (N // 128) * 2 * 128 * d * 2 + B * H * N * d * 2
    assert bench.ceiling_counts(synth.workload("T_b2h32n4096d128_bf16"))["l2_bytes"] == want
