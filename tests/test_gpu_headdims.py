"""Head dimensions beyond 64 and 128: every multiple of 8 up to 256, through
the four kernel widths (64, 128, 192, 256), against the oracle."""
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


def _inputs(seed, B, H, Nq, Nk, d, dtype):
    q = synth.tensor_bits(seed, (B, H, Nq, d), dtype)
    k = synth.tensor_bits(seed + 1, (B, H, Nk, d), dtype)
    v = synth.tensor_bits(seed + 2, (B, H, Nk, d), dtype)
    return q, k, v


CASES = [  # (d, dtype, mask, splits)
    (8, synth.FP16, 0, 1),
    (32, synth.BF16, 1, 1),
    (96, synth.FP16, 0, 1),
    (96, synth.BF16, 1, 3),
    (160, synth.BF16, 0, 1),
    (192, synth.FP16, 0, 1),
    (192, synth.BF16, 1, 1),
    (192, synth.FP16, 2, 3),
    (256, synth.BF16, 0, 1),
    (256, synth.FP16, 1, 1),
    (256, synth.BF16, 2, 1),
    (256, synth.BF16, 0, 3),
    (256, synth.FP16, 1, 4),
    (248, synth.BF16, 1, 1),
]


@pytest.mark.parametrize("d,dtype,mask,splits", CASES)
def test_head_dim(d, dtype, mask, splits):
    """Several 64/128-key tiles with a ragged tail, query tiles with a ragged
    tail; O is written into rows 8 elements wider than d whose padding holds
    a canary that must survive (columns beyond d are never stored)."""
    import torch
    import online_softmax_tiling_gb300 as fa
    B, H, Nq, Nk = 1, 2, 333, 397
    q, k, v = _inputs(400000 + 10 * d + mask, B, H, Nq, Nk, d, dtype)
    qd, kd, vd = (parity.to_device(x, dtype) for x in (q, k, v))
    store = torch.full((B, H, Nq, d + 8), -1000.0, dtype=qd.dtype, device="cuda")
    o, lse = fa.attention_forward_ex(qd, kd, vd, mask=mask, out=store[..., :d], num_splits=splits)
    assert fa.fa_check_device_status(None) == fa.FA_OK
    assert (store[..., d:] == -1000.0).all()
    parity.check_rows(q, k, v, dtype, mask, o, lse, f"d={d} mask={mask} splits={splits}")


@pytest.mark.parametrize("d", [192, 256])
@pytest.mark.parametrize("dtype", [synth.FP16, synth.BF16])
def test_wide_growing_keys_move_the_reference(d, dtype):
    """Key magnitudes that grow tile by tile, so the reference maximum moves
    and U is rescaled while the previous P.V may still be in flight."""
    B, H, N = 1, 2, 700
    q = synth.tensor_bits(611, (B, H, N, d), dtype)
    kf = synth.bits_to_float(synth.tensor_bits(612, (B, H, N, d), dtype), dtype).astype(np.float64)
    growth = 6.0 if dtype == synth.FP16 else 40.0
    kf *= (1.0 + growth * (np.arange(N) // 64) / 10.0)[None, None, :, None]
    k = synth.round_to_bits(kf, dtype)
    v = synth.tensor_bits(613, (B, H, N, d), dtype)
    for causal in (False, True):
        o, lse, ok = parity.run_gpu(q, k, v, dtype, 1.0 / math.sqrt(d), causal, guard=256)
        assert ok
        rows = np.arange(B * H * N, dtype=np.int64)
        o_ref, lse_ref, spread = parity.oracle_rows(q, k, v, dtype, 1.0 / math.sqrt(d), causal, rows)
        st = parity.compare(o.reshape(-1, d), lse.reshape(-1), o_ref, lse_ref, spread, dtype)
        parity.assert_within(st, f"growing keys d={d} causal={causal}", parity.WIDENED)


@pytest.mark.parametrize("d,causal", [(256, False), (256, True), (192, False)])
def test_wide_full_size_sampled(d, causal):
    """B=1, H=16, N=4096 in bf16 (the size the wide kernel is timed at); sampled rows."""
    B, H, N, dtype = 1, 16, 4096, synth.BF16
    q, k, v = _inputs(500000 + d + int(causal), B, H, N, N, d, dtype)
    o, lse, _ = parity.run_gpu(q, k, v, dtype, 1.0 / math.sqrt(d), causal)
    rows = synth.sample_rows(B * H, N, 1024, 77 + d)
    o_ref, lse_ref, spread = parity.oracle_rows(q, k, v, dtype, 1.0 / math.sqrt(d), causal, rows)
    st = parity.compare(o.reshape(-1, d)[rows], lse.reshape(-1)[rows], o_ref, lse_ref, spread, dtype)
    parity.assert_within(st, f"d={d} N=4096 causal={causal}")


@pytest.mark.parametrize("d", [96, 256])
@pytest.mark.parametrize("mask,fixture", [(0, "worked_example.txt"),
                                          (1, "worked_example_causal.txt"),
                                          (2, "worked_example_bottom_right.txt")])
def test_worked_example_embedded_wide(d, mask, fixture):
    """The printed 2-query / 4-key example ("先固定一个例子", Fig. 2-4, s = ln 2)
    zero-padded to d columns, with Nq = 2 and Nk = 4 as printed: O must be the
    fp16 rounding of the fixture's exact values, LSE within 1e-4."""
    import online_softmax_tiling_gb300 as fa
    from tests.golden import fixtures
    ex = fixtures.load("worked_example.txt")
    want = fixtures.load(fixture)
    dtype = synth.FP16
    q = np.zeros((1, 1, 2, d)); k = np.zeros((1, 1, 4, d)); v = np.zeros((1, 1, 4, d))
    q[0, 0, :, :2] = ex["Q"]
    k[0, 0, :, :2] = ex["K"]
    v[0, 0, :, :2] = ex["V"]
    qd, kd, vd = (parity.to_device(synth.round_to_bits(x, dtype), dtype) for x in (q, k, v))
    o, lse = fa.attention_forward_ex(qd, kd, vd, scale=math.log(2.0), mask=mask)
    assert fa.fa_check_device_status(None) == fa.FA_OK
    o = synth.bits_to_float(parity.from_device(o), dtype)[0, 0].astype(np.float64)
    want_o = synth.bits_to_float(synth.round_to_bits(want["O"][:2], dtype), dtype)
    np.testing.assert_array_equal(o[:, :2], want_o)
    np.testing.assert_array_equal(o[:, 2:], 0.0)
    np.testing.assert_allclose(lse.cpu().numpy()[0, 0], want["LSE"][:2], rtol=0, atol=1e-4)
