"""fa_fwd_ex: unequal query and key lengths, the three masks, strided tensors,
and split-KV on top, against the oracle."""
import math

import numpy as np
import pytest

import oracle
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


CASES = [  # (B, H, Nq, Nk, d, dtype, mask)
    (1, 2, 300, 700, 128, synth.BF16, 0),
    (1, 2, 300, 700, 128, synth.BF16, 1),
    (1, 2, 300, 700, 128, synth.BF16, 2),
    (2, 1, 700, 300, 64, synth.FP16, 1),
    (2, 1, 700, 300, 64, synth.FP16, 2),      # the first 400 queries see no key
    (1, 1, 1, 1000, 128, synth.FP16, 2),      # one query (decoding): sees every key
    (1, 3, 129, 50, 64, synth.BF16, 0),
    (1, 1, 513, 1000, 128, synth.FP16, 2),    # bottom-right diagonal across tile edges
]


@pytest.mark.parametrize("B,H,Nq,Nk,d,dtype,mask", CASES)
@pytest.mark.parametrize("splits", [1, 3])
def test_unequal_lengths_and_masks(B, H, Nq, Nk, d, dtype, mask, splits):
    import online_softmax_tiling_gb300 as fa
    seed = 300000 + Nq * 7 + Nk * 13 + d + mask
    q = synth.tensor_bits(seed, (B, H, Nq, d), dtype)
    k = synth.tensor_bits(seed + 1, (B, H, Nk, d), dtype)
    v = synth.tensor_bits(seed + 2, (B, H, Nk, d), dtype)
    qd, kd, vd = (parity.to_device(x, dtype) for x in (q, k, v))
    o, lse = fa.attention_forward_ex(qd, kd, vd, mask=mask, num_splits=splits)
    assert fa.fa_check_device_status(None) == fa.FA_OK
    parity.check_rows(q, k, v, dtype, mask, o, lse, f"Nq{Nq} Nk{Nk} mask{mask} splits{splits}")


def test_strided_bshd_views_in_and_out():
    """[B, N, H, d] storage (row stride H*d, head stride d) read and written in
    place, with LSE written into a padded buffer."""
    import torch
    import online_softmax_tiling_gb300 as fa
    B, H, N, d, dtype = 2, 3, 333, 128, synth.BF16
    q, k, v = (synth.tensor_bits(900 + i, (B, H, N, d), dtype) for i in range(3))
    bshd = [parity.to_device(x, dtype).permute(0, 2, 1, 3).contiguous() for x in (q, k, v)]
    qv, kv, vv = (t.permute(0, 2, 1, 3) for t in bshd)       # [B, H, N, d] views
    assert qv.stride() == (N * H * d, d, H * d, 1)
    o_store = torch.full((B, N, H, d), -1.0, dtype=qv.dtype, device="cuda")
    lse_store = torch.full((B, H, N + 5), -1.0, dtype=torch.float32, device="cuda")
    for mask in (0, 1):
        o, lse = fa.attention_forward_ex(qv, kv, vv, mask=mask, out=o_store.permute(0, 2, 1, 3),
                                         lse=lse_store[:, :, :N])
        assert fa.fa_check_device_status(None) == fa.FA_OK
        assert (lse_store[:, :, N:] == -1.0).all()           # padding untouched
        parity.check_rows(q, k, v, dtype, mask, o, lse, f"bshd mask{mask}")


def test_ex_matches_fa_fwd_bitwise_on_contiguous():
    import torch
    import online_softmax_tiling_gb300 as fa
    B, H, N, d, dtype = 1, 2, 1000, 64, synth.FP16
    q, k, v = (synth.tensor_bits(950 + i, (B, H, N, d), dtype) for i in range(3))
    qd, kd, vd = (parity.to_device(x, dtype) for x in (q, k, v))
    for causal in (False, True):
        o1, l1 = fa.attention_forward(qd, kd, vd, causal=causal)
        o2, l2 = fa.attention_forward_ex(qd, kd, vd, mask=int(causal))
        assert torch.equal(o1, o2) and torch.equal(l1, l2)
