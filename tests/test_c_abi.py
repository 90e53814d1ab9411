"""The boundary from C: a C99 program includes include/fa.h, links the
library and the CUDA runtime, and runs fa_fwd; its output is checked against
the oracle (on a GPU) after it compiles and links (everywhere)."""
import math
import os
import subprocess

import numpy as np
import pytest

import online_softmax_tiling_gb300 as fa
from online_softmax_tiling_gb300 import synth
from tests.c_abi import build as cbuild


@pytest.fixture(scope="module")
def exe(tmp_path_factory):
    if not os.path.exists(fa.LIBRARY):
        from online_softmax_tiling_gb300 import build
        build.build()
    return cbuild.build(str(tmp_path_factory.mktemp("c_abi")))


def test_c_caller_compiles_and_links(exe):
    assert os.access(exe, os.X_OK)


@pytest.mark.gpu
@pytest.mark.parametrize("causal,dtype", [(0, synth.FP16), (1, synth.BF16)])
def test_c_caller_matches_oracle(exe, tmp_path, causal, dtype):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from tests import parity
    B, H, N, d = 1, 3, 500, 128
    scale = 1.0 / math.sqrt(d)
    q, k, v = (synth.tensor_bits(990000 + 10 * causal + i, (B, H, N, d), dtype) for i in range(3))
    src, dst = tmp_path / "in.bin", tmp_path / "out.bin"
    with open(src, "wb") as f:
        f.write(np.array([B, H, N, d, causal, dtype], dtype=np.int32).tobytes())
        f.write(np.array([scale], dtype=np.float32).tobytes())
        for x in (q, k, v):
            f.write(np.ascontiguousarray(x, dtype=np.uint16).tobytes())
    r = subprocess.run([exe, str(src), str(dst)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    raw = np.fromfile(dst, dtype=np.uint8)
    n = B * H * N * d
    o = raw[:2 * n].view(np.uint16).reshape(B * H * N, d)
    lse = raw[2 * n:].view(np.float32)
    rows = np.arange(B * H * N, dtype=np.int64)
    o_ref, lse_ref, spread = parity.oracle_rows(q, k, v, dtype, scale, bool(causal), rows)
    st = parity.compare(o, lse, o_ref, lse_ref, spread, dtype)
    parity.assert_within(st, f"C caller causal={causal}")
