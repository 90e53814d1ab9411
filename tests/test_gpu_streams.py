"""The library on several streams and inside CUDA graphs: two independent
problems enqueued on two streams at once, and fa_fwd / split-KV captured in
a graph and replayed on new inputs copied into the captured buffers."""
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


def _problem(seed, B, H, N, d, dtype):
    return tuple(synth.tensor_bits(seed + i, (B, H, N, d), dtype) for i in range(3))


def test_two_streams_at_once():
    import torch
    import online_softmax_tiling_gb300 as fa
    dtype = synth.BF16
    probs = [_problem(970000, 2, 4, 1000, 128, dtype), _problem(970100, 1, 8, 777, 64, dtype)]
    causal = [False, True]
    dev = [tuple(parity.to_device(x, dtype) for x in pr) for pr in probs]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = []
    for (qd, kd, vd), c, st in zip(dev, causal, streams):
        with torch.cuda.stream(st):
            outs.append(fa.attention_forward(qd, kd, vd, causal=c, stream=st))
    torch.cuda.synchronize()
    assert fa.fa_check_device_status(None) == fa.FA_OK
    for (q, k, v), c, (o, lse) in zip(probs, causal, outs):
        parity.check_rows(q, k, v, dtype, int(c), o, lse, f"stream causal={c}")


@pytest.mark.parametrize("splits", [1, 4])
def test_graph_capture_and_replay(splits):
    import torch
    import online_softmax_tiling_gb300 as fa
    B, H, N, d, dtype = 1, 2, 1000, 128, synth.FP16
    tdt = torch.float16
    first = _problem(980000, B, H, N, d, dtype)
    second = _problem(980100, B, H, N, d, dtype)
    q, k, v = (torch.empty((B, H, N, d), dtype=tdt, device="cuda") for _ in range(3))
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    for dst, src in zip((q, k, v), first):
        dst.copy_(parity.to_device(src, dtype))
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        # warm-up outside the capture (the library sets kernel attributes once)
        fa.attention_forward(q, k, v, causal=True, out=o, lse=lse, stream=stream,
                             num_splits=splits)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        fa.attention_forward(q, k, v, causal=True, out=o, lse=lse,
                             stream=torch.cuda.current_stream(), num_splits=splits)
    for inputs in (first, second):
        for dst, src in zip((q, k, v), inputs):
            dst.copy_(parity.to_device(src, dtype))
        o.fill_(0)
        graph.replay()
        torch.cuda.synchronize()
        assert fa.fa_check_device_status(None) == fa.FA_OK
        parity.check_rows(*inputs, dtype, 1, o, lse, f"graph replay splits={splits}")
