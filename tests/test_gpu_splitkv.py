"""Split-KV ("CUDA 算子工程" 14.7.1): partial results over key ranges merged by
their log-sum-exps, against the oracle and against the one-launch path."""
import math

import numpy as np
import pytest

from online_softmax_tiling_gb300 import synth
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from online_softmax_tiling_gb300 import build
    build.build()
    yield


CASES = [  # (B, H, N, d, dtype, causal, num_splits); 0 = the library's choice
    (1, 1, 4096, 64, synth.FP16, False, 0),
    (1, 1, 4096, 64, synth.FP16, False, 8),
    (1, 2, 1000, 128, synth.BF16, True, 3),
    (1, 2, 1000, 128, synth.BF16, False, 7),
    (2, 1, 300, 64, synth.BF16, True, 4),      # more splits than some blocks have tiles
    (1, 1, 129, 128, synth.FP16, True, 32),    # mostly empty ranges
    (1, 1, 64, 64, synth.FP16, False, 2),      # one key tile, one empty range
    (1, 3, 2048, 128, synth.FP16, True, 5),
    (1, 8, 4000, 128, synth.BF16, True, 0),    # causal, one wave of blocks: the library splits it
]


@pytest.mark.parametrize("B,H,N,d,dtype,causal,splits", CASES)
def test_splitkv_matches_oracle(B, H, N, d, dtype, causal, splits):
    seed = 200000 + 31 * N + d + 7 * dtype + int(causal) + 101 * splits
    q = synth.tensor_bits(seed, (B, H, N, d), dtype)
    k = synth.tensor_bits(seed + 1, (B, H, N, d), dtype)
    v = synth.tensor_bits(seed + 2, (B, H, N, d), dtype)
    scale = 1.0 / math.sqrt(d)
    o, lse, guards = parity.run_gpu(q, k, v, dtype, scale, causal, guard=4096, num_splits=splits)
    assert guards, "write outside O or LSE"
    rows = np.arange(B * H * N, dtype=np.int64)
    if rows.size > 4096:
        rows = synth.sample_rows(B * H, N, 3000, seed)
    o_ref, lse_ref, spread = parity.oracle_rows(q, k, v, dtype, scale, causal, rows)
    st = parity.compare(o.reshape(-1, d)[rows], lse.reshape(-1)[rows], o_ref, lse_ref, spread, dtype)
    parity.assert_within(st, f"split {splits} B{B}H{H}N{N}d{d}")


def test_splitkv_agrees_with_one_launch():
    B, H, N, d, dtype = 1, 4, 2048, 128, synth.BF16
    q, k, v = (synth.tensor_bits(777 + i, (B, H, N, d), dtype) for i in range(3))
    scale = 1.0 / math.sqrt(d)
    for causal in (False, True):
        o1, l1, _ = parity.run_gpu(q, k, v, dtype, scale, causal)
        o2, l2, _ = parity.run_gpu(q, k, v, dtype, scale, causal, num_splits=6)
        a = synth.bits_to_float(o1, dtype).astype(np.float64)
        b = synth.bits_to_float(o2, dtype).astype(np.float64)
        assert np.abs(a - b).max() <= 2 * 2.0 ** -8 * max(1.0, np.abs(a).max())
        np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-4)
