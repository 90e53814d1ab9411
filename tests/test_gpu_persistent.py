"""The persistent grid: more query blocks ("units") than SMs, so every CTA
walks several of them and the barrier phases, ring positions and TMEM
hand-offs run on from one unit to the next.  Every row is compared with the
oracle; the shapes mix unit lengths (causal masks), units whose first query
tile sees no key (bottom-right mask with more queries than keys), split-KV
ranges and strided views."""
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


def _sms():
    import torch
    return torch.cuda.get_device_properties(0).multi_processor_count


CASES = [  # (B, H, Nq, Nk, d, dtype, mask, splits)
    (4, 48, 300, 700, 64, synth.FP16, 2, 1),      # 384 units of two lengths
    (3, 40, 700, 300, 128, synth.BF16, 2, 1),     # 360 units; the first 400 queries see no key
    (2, 100, 600, 600, 128, synth.FP16, 1, 1),    # 600 causal units, longest first
    (2, 60, 900, 900, 64, synth.BF16, 1, 3),      # 1440 units: causal, three key ranges each
    (1, 200, 256, 256, 128, synth.BF16, 0, 1),    # 200 units of two key tiles
    (2, 40, 700, 300, 256, synth.BF16, 2, 1),     # wide heads: 480 units, some see no key
    (1, 60, 500, 500, 192, synth.FP16, 1, 2),     # wide heads: 480 causal units, two key ranges
]


@pytest.mark.parametrize("B,H,Nq,Nk,d,dtype,mask,splits", CASES)
def test_many_units_per_cta(B, H, Nq, Nk, d, dtype, mask, splits):
    import online_softmax_tiling_gb300 as fa
    block = 256 if d <= 128 else 128  # query rows per unit
    units = B * H * ((Nq + block - 1) // block) * splits
    assert units > _sms(), "the shape must give some CTA more than one unit"
    seed = 710000 + 11 * H + Nq + 3 * Nk + d + 5 * mask + splits
    q = synth.tensor_bits(seed, (B, H, Nq, d), dtype)
    k = synth.tensor_bits(seed + 1, (B, H, Nk, d), dtype)
    v = synth.tensor_bits(seed + 2, (B, H, Nk, d), dtype)
    qd, kd, vd = (parity.to_device(x, dtype) for x in (q, k, v))
    o, lse = fa.attention_forward_ex(qd, kd, vd, mask=mask, num_splits=splits)
    assert fa.fa_check_device_status(None) == fa.FA_OK
    parity.check_rows(q, k, v, dtype, mask, o, lse,
                      f"B{B} H{H} Nq{Nq} Nk{Nk} d{d} mask{mask} splits{splits}")


def test_one_unit_more_than_sms():
    """SMs + 1 units: one CTA takes a second unit in the reversed second round."""
    import online_softmax_tiling_gb300 as fa
    H, N, d, dtype = _sms() + 1, 256, 64, synth.FP16
    q, k, v = (synth.tensor_bits(720000 + i, (1, H, N, d), dtype) for i in range(3))
    qd, kd, vd = (parity.to_device(x, dtype) for x in (q, k, v))
    o, lse = fa.attention_forward(qd, kd, vd, scale=1.0 / math.sqrt(d), causal=False)
    assert fa.fa_check_device_status(None) == fa.FA_OK
    parity.check_rows(q, k, v, dtype, 0, o, lse, f"H{H}")


def test_many_units_strided_views():
    """[B, N, H, d] storage viewed as [B, H, N, d], 400 causal units."""
    import torch
    import online_softmax_tiling_gb300 as fa
    B, H, N, d, dtype = 2, 50, 1000, 128, synth.BF16
    q, k, v = (synth.tensor_bits(730000 + i, (B, H, N, d), dtype) for i in range(3))
    bshd = [parity.to_device(np.ascontiguousarray(x.transpose(0, 2, 1, 3)), dtype) for x in (q, k, v)]
    qv, kv, vv = (t.permute(0, 2, 1, 3) for t in bshd)
    o_store = torch.zeros((B, N, H, d), dtype=qv.dtype, device="cuda")
    ov = o_store.permute(0, 2, 1, 3)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    fa.attention_forward_ex(qv, kv, vv, mask=1, out=ov, lse=lse)
    assert fa.fa_check_device_status(None) == fa.FA_OK
    parity.check_rows(q, k, v, dtype, 1, ov, lse, "strided causal")


ONE_TILE_CASES = [  # (B, H, Nq, Nk, d, dtype, mask, splits): 256-row blocks fit one wave
    (1, 76, 512, 512, 128, synth.BF16, 1, 1),     # 152 blocks -> 304 one-tile units
    (1, 50, 520, 520, 64, synth.FP16, 1, 1),      # 150 blocks -> 250 units, ragged tail
    (1, 60, 400, 600, 128, synth.BF16, 2, 1),     # bottom-right, more keys than queries
    (1, 50, 700, 300, 128, synth.FP16, 2, 1),     # bottom-right: the first 400 queries see no key
    (1, 36, 900, 900, 128, synth.BF16, 1, 2),     # one-tile units in two key ranges
]


@pytest.mark.parametrize("B,H,Nq,Nk,d,dtype,mask,splits", ONE_TILE_CASES)
def test_many_one_tile_units_per_cta(B, H, Nq, Nk, d, dtype, mask, splits):
    """Causal grids whose two-tile blocks fit in one wave run one 128-row
    query tile per unit (twice as many units); here more than there are SMs."""
    import online_softmax_tiling_gb300 as fa
    blocks = B * H * ((Nq + 255) // 256)
    units = B * H * ((Nq + 127) // 128) * splits
    if blocks > _sms():
        pytest.skip("the case assumes the one-tile kernel serves it (blocks fit in one wave)")
    assert units > _sms(), "the shape must give some CTA more than one unit"
    seed = 740000 + 11 * H + Nq + 3 * Nk + d + 5 * mask + splits
    q = synth.tensor_bits(seed, (B, H, Nq, d), dtype)
    k = synth.tensor_bits(seed + 1, (B, H, Nk, d), dtype)
    v = synth.tensor_bits(seed + 2, (B, H, Nk, d), dtype)
    qd, kd, vd = (parity.to_device(x, dtype) for x in (q, k, v))
    o, lse = fa.attention_forward_ex(qd, kd, vd, mask=mask, num_splits=splits)
    assert fa.fa_check_device_status(None) == fa.FA_OK
    parity.check_rows(q, k, v, dtype, mask, o, lse,
                      f"one-tile B{B} H{H} Nq{Nq} Nk{Nk} d{d} mask{mask} splits{splits}")
