"""Every compiled kernel instantiation runs in one process and matches the
oracle: 4 widths x 2 types x (no mask, causal) x (plain, split-KV) of the
fused path, and 2 widths x 2 types of the step-by-step baseline."""
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


def test_every_instantiation_launches_and_matches():
    import online_softmax_tiling_gb300 as fa
    B, H, N = 1, 1, 200
    n = 0
    for d in (64, 128, 192, 256):
        for dtype in (synth.FP16, synth.BF16):
            q, k, v = (synth.tensor_bits(810000 + d + 7 * dtype + i, (B, H, N, d), dtype)
                       for i in range(3))
            qd, kd, vd = (parity.to_device(x, dtype) for x in (q, k, v))
            for mask in (0, 1):
                for splits in (1, 2):
                    o, lse = fa.attention_forward_ex(qd, kd, vd, mask=mask, num_splits=splits)
                    assert fa.fa_check_device_status(None) == fa.FA_OK
                    parity.check_rows(q, k, v, dtype, mask, o, lse,
                                      f"d={d} dtype={dtype} mask={mask} splits={splits}")
                    n += 1
            if d <= 128:
                o, lse = fa.naive_attention_forward(qd, kd, vd, scale=1.0 / math.sqrt(d))
                assert fa.fa_check_device_status(None) == fa.FA_OK
                assert np.isfinite(synth.bits_to_float(parity.from_device(o), dtype)).all()
                n += 1
    assert n == 36
