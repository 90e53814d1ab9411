"""The step-by-step baseline (S and P in HBM) against the oracle.

It stores S and P in the 16-bit input type, as the traffic count of
"CUDA 算子工程" ch. 14, section 14.2 assumes (2 bytes per element), so its
error is larger than the fused kernel's and its bound is derived here from
that arithmetic (u = unit roundoff of the 16-bit type):
  * S_j rounded: |dS_j| <= u |S_j|, so every weight exp(S_j - m) / l moves
    by a factor within exp(+-2 u max_j |S_j|);
  * P_j rounded once more (relative u), not renormalised;
  * so |dO_c| <= half an ulp of O + (e^{2 u Smax} (1 + u) - 1) sum_j P_j |v_jc|
    (+ fp32 accumulation), with sum_j P_j |v_jc| <= spread_c + |O_c|;
  * |dLSE| <= u Smax (+ fp32 rounding).
"""
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


def _smax(q, k, dtype, scale, causal, rows):
    """max_j |s q_i . k_j| over each row's visible keys (fp64 from the bits)."""
    B, H, N, d = q.shape
    qf = synth.bits_to_float(q, dtype).astype(np.float64).reshape(B * H, N, d)
    kf = synth.bits_to_float(k, dtype).astype(np.float64).reshape(B * H, N, d)
    out = np.empty(rows.size)
    for n, r in enumerate(rows):
        bh, i = divmod(int(r), N)
        nv = i + 1 if causal else N
        out[n] = np.abs(scale * (kf[bh, :nv] @ qf[bh, i])).max()
    return out


def _check(q, k, v, dtype, scale, causal, o_bits, lse, rows, label):
    d = q.shape[-1]
    o_ref, lse_ref, spread = parity.oracle_rows(q, k, v, dtype, scale, causal, rows)
    u = parity.UNIT_ROUNDOFF[dtype]
    smax = _smax(q, k, dtype, scale, causal, rows)
    o = synth.bits_to_float(o_bits.reshape(-1, d)[rows], dtype).astype(np.float64)
    fac = (np.exp(2 * u * smax) * (1 + u) - 1)[:, None]
    bound = parity.half_ulp(np.maximum(np.abs(o), np.abs(o_ref)), dtype) + \
        fac * (spread + np.abs(o_ref)) + 1e-5 * (np.abs(o_ref) + spread)
    err = np.abs(o - o_ref)
    assert np.isfinite(o).all(), label
    assert (err <= bound).all(), f"{label}: worst excess {(err - bound).max():.3g}"
    lerr = np.abs(lse.reshape(-1)[rows].astype(np.float64) - lse_ref)
    assert (lerr <= u * smax + 2e-6 * np.maximum(1, np.abs(lse_ref))).all(), \
        f"{label}: LSE {lerr.max():.3g}"


CASES = [  # (B, H, N, d, dtype, causal)
    (1, 1, 128, 64, synth.FP16, False),
    (1, 2, 1000, 64, synth.FP16, False),
    (2, 1, 512, 64, synth.BF16, True),
    (1, 1, 1024, 128, synth.BF16, True),
    (1, 2, 392, 128, synth.FP16, False),
]


@pytest.mark.parametrize("B,H,N,d,dtype,causal", CASES)
def test_naive_matches_oracle(B, H, N, d, dtype, causal):
    import online_softmax_tiling_gb300 as fa
    seed = 700000 + N + d + int(causal)
    q, k, v = (synth.tensor_bits(seed + i, (B, H, N, d), dtype) for i in range(3))
    qd, kd, vd = (parity.to_device(x, dtype) for x in (q, k, v))
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.naive_attention_forward(qd, kd, vd, scale=scale, causal=causal)
    assert fa.fa_check_device_status(None) == fa.FA_OK
    rows = np.arange(B * H * N, dtype=np.int64)
    _check(q, k, v, dtype, scale, causal, parity.from_device(o), lse.cpu().numpy(), rows,
           f"naive N={N} d={d} causal={causal}")


def test_naive_on_the_pages_traffic_shape():
    """C2 (B=1, H=1, N=4096, d=64, fp16): the shape of the pages' traffic count."""
    import online_softmax_tiling_gb300 as fa
    w = synth.workload("C2")
    q, k, v = synth.make_inputs(w)
    qd, kd, vd = (parity.to_device(x, w.dtype) for x in (q, k, v))
    o, lse = fa.naive_attention_forward(qd, kd, vd, scale=w.scale, causal=w.causal)
    assert fa.fa_check_device_status(None) == fa.FA_OK
    rows = synth.sample_rows(1, w.N, 1024, 91)
    _check(q, k, v, w.dtype, w.scale, w.causal, parity.from_device(o), lse.cpu().numpy(), rows,
           "naive C2")
