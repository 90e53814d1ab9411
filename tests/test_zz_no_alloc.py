"""The split-KV entry point for callers that cannot allocate device memory.

A plugin whose host framework owns all device memory, or a latency-critical
path that cannot take cudaMalloc's implicit synchronisation, cannot provide a
workspace.  fa_fwd_splitkv_noalloc keeps the partials in a fixed array inside
the library instead.  Its output must match the workspace entry point's
(fa_fwd_splitkv) within the tolerances the other tests use, on calls made one
after the other (the array keeps the previous call's contents).  Collected
last, and independent of every other test.
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


def _run(entry, q_bits, k_bits, v_bits, dtype, scale, causal, splits):
    import torch
    import online_softmax_tiling_gb300 as fa
    B, H, N, d = q_bits.shape
    q, k, v = (parity.to_device(x, dtype) for x in (q_bits, k_bits, v_bits))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    args = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d,
            scale, int(causal), dtype, splits)
    if entry == "workspace":
        nbytes = fa.fa_splitkv_workspace_size(B, H, N, d, splits)
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        st = fa.fa_fwd_splitkv(*args, ws.data_ptr(), nbytes, s)
    else:
        st = fa.fa_fwd_splitkv_noalloc(*args, s)
    assert st == fa.FA_OK, fa.fa_status_string(st)
    assert fa.fa_check_device_status(s) == fa.FA_OK
    return parity.from_device(o), lse.cpu().numpy()


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls():
    cases = [((1, 1, 4096, 64), synth.FP16, False, 8, 61),
             ((1, 2, 1000, 128), synth.BF16, True, 4, 62)]
    for shape, dtype, causal, splits, seed in cases:     # two calls in a row
        q, k, v = (synth.tensor_bits(seed * 10 + i, shape, dtype) for i in range(3))
        scale = 1.0 / math.sqrt(shape[-1])
        o_ws, l_ws = _run("workspace", q, k, v, dtype, scale, causal, splits)
        o_na, l_na = _run("noalloc", q, k, v, dtype, scale, causal, splits)
        a = synth.bits_to_float(o_ws, dtype).astype(np.float64)
        b = synth.bits_to_float(o_na, dtype).astype(np.float64)
        assert np.isfinite(b).all() and np.isfinite(l_na).all()
        assert np.abs(a - b).max() <= parity.MAX_EXCESS
        assert np.abs(a - b).mean() <= parity.MEAN_EXCESS
        rel = np.abs(l_ws - l_na) / np.maximum(1.0, np.abs(l_ws))
        assert rel.max() <= parity.LSE_REL


def test_noalloc_rejects_requests_beyond_its_array():
    import online_softmax_tiling_gb300 as fa
    B, H, N, d, splits = 8, 16, 4096, 128, 8
    assert fa.fa_splitkv_workspace_size(B, H, N, d, splits) > fa.FA_NOALLOC_SCRATCH_BYTES
    A = 0x10000   # never dereferenced: the request is refused before any launch
    st = fa.fa_fwd_splitkv_noalloc(A, A + 0x1000, A + 0x2000, A + 0x3000, A + 0x4000, B, H, N, d,
                                   0.1, 0, fa.FA_BF16, splits, None)
    assert st == fa.FA_ERR_UNSUPPORTED
