"""Sizes at the edges of what the kernels are built for, checked on sampled
rows against the oracle: a 131072-long sequence (512 query blocks of one
head, 1024 key tiles per row), 4096 heads of 128 rows, and one query row
against 262144 keys through split-KV."""
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


def _rows(BH, N, count, seed):
    rows = synth.sample_rows(BH, N, count, seed)
    last = np.arange(max(0, BH * N - 8), BH * N, dtype=np.int64)      # the longest causal rows
    return np.unique(np.concatenate([rows, last]))


@pytest.mark.parametrize("causal", [False, True])
def test_long_sequence(causal):
    B, H, N, d, dtype = 1, 1, 131072, 128, synth.BF16
    q, k, v = (synth.tensor_bits(920000 + i + 10 * int(causal), (B, H, N, d), dtype) for i in range(3))
    o, lse, ok = parity.run_gpu(q, k, v, dtype, 1.0 / math.sqrt(d), causal, guard=64)
    assert ok
    rows = _rows(1, N, 160, 11 + int(causal))
    o_ref, lse_ref, spread = parity.oracle_rows(q, k, v, dtype, 1.0 / math.sqrt(d), causal, rows)
    st = parity.compare(o.reshape(-1, d)[rows], lse.reshape(-1)[rows], o_ref, lse_ref, spread, dtype)
    parity.assert_within(st, f"N=131072 causal={causal}")


def test_many_heads():
    B, H, N, d, dtype = 64, 64, 128, 64, synth.FP16
    q, k, v = (synth.tensor_bits(930000 + i, (B, H, N, d), dtype) for i in range(3))
    o, lse, ok = parity.run_gpu(q, k, v, dtype, 0.125, True, guard=64)
    assert ok
    rows = _rows(B * H, N, 2048, 13)
    o_ref, lse_ref, spread = parity.oracle_rows(q, k, v, dtype, 0.125, True, rows)
    st = parity.compare(o.reshape(-1, d)[rows], lse.reshape(-1)[rows], o_ref, lse_ref, spread, dtype)
    parity.assert_within(st, "4096 heads")


def test_one_query_against_a_long_key_sequence():
    import online_softmax_tiling_gb300 as fa
    B, H, Nq, Nk, d, dtype = 1, 8, 1, 262144, 128, synth.BF16
    q = synth.tensor_bits(940000, (B, H, Nq, d), dtype)
    k = synth.tensor_bits(940001, (B, H, Nk, d), dtype)
    v = synth.tensor_bits(940002, (B, H, Nk, d), dtype)
    qd, kd, vd = (parity.to_device(x, dtype) for x in (q, k, v))
    args = fa.fa_fwd_args()
    args.B, args.H, args.Nq, args.Nk, args.d = B, H, Nq, Nk, d
    splits = fa.fa_splitkv_num_splits_ex(args)
    assert splits > 1                     # 8 one-row blocks on a GPU of 100+ SMs
    for mask in (0, 2):
        o, lse = fa.attention_forward_ex(qd, kd, vd, mask=mask, num_splits=0)
        assert fa.fa_check_device_status(None) == fa.FA_OK
        parity.check_rows(q, k, v, dtype, mask, o, lse, f"decode Nk=262144 mask={mask}")
