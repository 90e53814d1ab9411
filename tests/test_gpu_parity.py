"""GPU parity: the CUDA path, called through the C ABI, against the oracle.

Full element-by-element comparison at sizes the oracle finishes in seconds
(several 128-row tiles plus ragged tails), and sampled rows at the full sizes
of every workload in the configuration the benchmark times.  Tolerances are
those of tests/parity.py.
"""
import math

import numpy as np
import pytest

import oracle
from online_softmax_tiling_gb300 import synth
from tests import parity
from tests.golden import fixtures

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from online_softmax_tiling_gb300 import build
    build.build()
    yield


def _embed(mat, n, d):
    out = np.zeros((n, d))
    out[: mat.shape[0], : mat.shape[1]] = mat
    return out


@pytest.mark.parametrize("causal", [False, True])
def test_worked_example_embedded(causal):
    """The printed 2-query, 4-key, d=2 example (Fig. 2-12), zero-padded to d=64, fp16."""
    ex = fixtures.load("worked_example.txt")
    want = fixtures.load("worked_example_causal.txt" if causal else "worked_example.txt")
    N, d = 4, 64
    q = synth.round_to_bits(_embed(ex["Q"], N, d), synth.FP16)[None, None]
    k = synth.round_to_bits(_embed(ex["K"], N, d), synth.FP16)[None, None]
    v = synth.round_to_bits(_embed(ex["V"], N, d), synth.FP16)[None, None]
    o, lse, _ = parity.run_gpu(q, k, v, synth.FP16, math.log(2.0), causal)
    o = synth.bits_to_float(o[0, 0], synth.FP16).astype(np.float64)
    exp_o = synth.bits_to_float(synth.round_to_bits(want["O"], synth.FP16), synth.FP16)
    np.testing.assert_array_equal(o[:2, :2], exp_o)            # fp16 RNE of 7/8, 3/4, 4/3, 1/3
    np.testing.assert_array_equal(o[:2, 2:], 0.0)
    np.testing.assert_allclose(lse[0, 0, :2], want["LSE"], rtol=0, atol=1e-4)


CASES = [  # (B, H, N, d, dtype, causal): several tiles, ragged tails, degenerate sizes
    (1, 1, 1, 64, synth.FP16, False),
    (1, 1, 1, 128, synth.BF16, True),
    (1, 2, 2, 64, synth.BF16, True),
    (2, 1, 63, 64, synth.FP16, True),
    (1, 2, 64, 128, synth.FP16, False),
    (1, 1, 65, 64, synth.BF16, False),
    (1, 1, 127, 128, synth.BF16, True),
    (1, 1, 128, 64, synth.FP16, True),
    (1, 1, 129, 128, synth.FP16, True),
    (2, 3, 300, 64, synth.FP16, False),
    (2, 3, 300, 64, synth.BF16, True),
    (2, 3, 300, 128, synth.FP16, True),
    (2, 3, 300, 128, synth.BF16, False),
    (1, 2, 517, 128, synth.BF16, True),
    (1, 1, 1000, 64, synth.FP16, True),
]


@pytest.mark.parametrize("B,H,N,d,dtype,causal", CASES)
def test_full_comparison_small(B, H, N, d, dtype, causal):
    seed = 100000 + 97 * N + d + 7 * dtype + int(causal)
    q = synth.tensor_bits(seed, (B, H, N, d), dtype)
    k = synth.tensor_bits(seed + 1, (B, H, N, d), dtype)
    v = synth.tensor_bits(seed + 2, (B, H, N, d), dtype)
    scale = 1.0 / math.sqrt(d)
    o, lse, guards = parity.run_gpu(q, k, v, dtype, scale, causal, guard=4096)
    assert guards, "write outside O or LSE"
    rows = np.arange(B * H * N, dtype=np.int64)
    o_ref, lse_ref, spread = parity.oracle_rows(q, k, v, dtype, scale, causal, rows)
    st = parity.compare(o.reshape(-1, d), lse.reshape(-1), o_ref, lse_ref, spread, dtype)
    parity.assert_within(st, f"B{B}H{H}N{N}d{d}")


def test_wide_score_range_rescales():
    """Scores spanning >> 2^8 in weight units force the running-maximum moves."""
    B, H, N, d, dtype = 1, 2, 700, 128, synth.BF16
    q = synth.tensor_bits(501, (B, H, N, d), dtype, mult=3.0)
    k = synth.tensor_bits(502, (B, H, N, d), dtype, mult=3.0)
    v = synth.tensor_bits(503, (B, H, N, d), dtype)
    scale = 1.0 / math.sqrt(d)
    for causal in (False, True):
        o, lse, _ = parity.run_gpu(q, k, v, dtype, scale, causal)
        rows = np.arange(B * H * N, dtype=np.int64)
        o_ref, lse_ref, spread = parity.oracle_rows(q, k, v, dtype, scale, causal, rows)
        st = parity.compare(o.reshape(-1, d), lse.reshape(-1), o_ref, lse_ref, spread, dtype)
        parity.assert_within(st, f"wide causal={causal}", parity.WIDENED)


@pytest.mark.parametrize("dtype", [synth.FP16, synth.BF16])
@pytest.mark.parametrize("causal", [False, True])
def test_growing_keys_move_the_reference(dtype, causal):
    """Key magnitudes that grow tile by tile: later tiles' weights overflow the
    bound against the stale reference, so the maximum is re-taken, U is
    rescaled and the weights recomputed."""
    B, H, N, d = 1, 2, 1000, 128
    q = synth.tensor_bits(601, (B, H, N, d), dtype)
    kf = synth.bits_to_float(synth.tensor_bits(602, (B, H, N, d), dtype), dtype).astype(np.float64)
    growth = 6.0 if dtype == synth.FP16 else 40.0
    kf *= (1.0 + growth * (np.arange(N) // 128) / 7.0)[None, None, :, None]
    k = synth.round_to_bits(kf, dtype)
    v = synth.tensor_bits(603, (B, H, N, d), dtype)
    scale = 1.0 / math.sqrt(d)
    o, lse, _ = parity.run_gpu(q, k, v, dtype, scale, causal)
    rows = np.arange(B * H * N, dtype=np.int64)
    o_ref, lse_ref, spread = parity.oracle_rows(q, k, v, dtype, scale, causal, rows)
    st = parity.compare(o.reshape(-1, d), lse.reshape(-1), o_ref, lse_ref, spread, dtype)
    parity.assert_within(st, f"growing keys dtype={dtype} causal={causal}", parity.WIDENED)


@pytest.mark.parametrize("dtype", [synth.FP16, synth.BF16])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_key_halves_move_the_reference(dtype, d, causal):
    """Key magnitudes that grow every 64 keys: the weights of a tile's first
    half may pass against the running reference while those of its second
    half overflow the bound after the first half went to the tensor core, so
    U absorbs the first half, is rescaled, and the second half is recomputed
    (tests/test_softmax_routes.py checks that these inputs take that route)."""
    q, k, v = parity.keys_growing_by_half(dtype, d)
    B, H, N, _ = q.shape
    scale = 1.0 / math.sqrt(d)
    o, lse, guards = parity.run_gpu(q, k, v, dtype, scale, causal, guard=4096)
    assert guards, "write outside O or LSE"
    rows = np.arange(B * H * N, dtype=np.int64)
    o_ref, lse_ref, spread = parity.oracle_rows(q, k, v, dtype, scale, causal, rows)
    st = parity.compare(o.reshape(-1, d), lse.reshape(-1), o_ref, lse_ref, spread, dtype)
    parity.assert_within(st, f"key halves dtype={dtype} d={d} causal={causal}", parity.WIDENED)


_INPUTS = {}


def _workload_inputs(name):
    if name not in _INPUTS:
        _INPUTS.clear()
        w = synth.workload(name)
        _INPUTS[name] = (w, *synth.make_inputs(w))
    return _INPUTS[name]


@pytest.mark.parametrize("name", ["C1", "C2", "C3", "C4", "C5", "C5r", "T_b2h32n4096d128_bf16",
                                  "T_b2h32n4096d128_fp16"])
def test_workload_full_size_sampled(name):
    """Each workload at its full size, as the benchmark runs it; sampled rows vs the oracle."""
    w, q, k, v = _workload_inputs(name)
    o, lse, _ = parity.run_gpu(q, k, v, w.dtype, w.scale, w.causal)
    BH = w.B * w.H
    rows = synth.sample_rows(BH, w.N, 1536 if w.N * w.d > 1 << 20 else 4096, w.seed_base + 9)
    o_ref, lse_ref, spread = parity.oracle_rows(q, k, v, w.dtype, w.scale, w.causal, rows)
    st = parity.compare(o.reshape(-1, w.d)[rows], lse.reshape(-1)[rows], o_ref, lse_ref, spread,
                        w.dtype)
    print(name, st)
    parity.assert_within(st, name, parity.gate_for(w))
    # every output is finite, and every row's weights sum to one implies
    # min_j v <= O <= max_j v per column: check the bound on all rows cheaply
    o_all = synth.bits_to_float(o, w.dtype)
    assert np.isfinite(o_all).all() and np.isfinite(lse).all()
    vmin = synth.bits_to_float(v, w.dtype).min(axis=2, keepdims=True)
    vmax = synth.bits_to_float(v, w.dtype).max(axis=2, keepdims=True)
    assert (o_all >= vmin - 1e-2).all() and (o_all <= vmax + 1e-2).all()


def test_repeatable_bitwise():
    w = synth.workload("C3")
    q = synth.tensor_bits(11, (1, 4, 1024, 64), w.dtype)
    k = synth.tensor_bits(12, (1, 4, 1024, 64), w.dtype)
    v = synth.tensor_bits(13, (1, 4, 1024, 64), w.dtype)
    a = parity.run_gpu(q, k, v, w.dtype, w.scale, True)
    b = parity.run_gpu(q, k, v, w.dtype, w.scale, True)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_bounded_wait_reports_timeout_and_context_survives():
    """A wait that nothing will satisfy (the loader skips the first key tile)
    runs out after its limit; the kernel reports FA_ERR_TIMEOUT and exits, and
    the next normal launch on the same context is correct."""
    import torch
    import online_softmax_tiling_gb300 as fa
    B, H, N, d, dtype = 1, 1, 256, 64, synth.FP16
    q_bits = synth.tensor_bits(71, (B, H, N, d), dtype)
    q = parity.to_device(q_bits, dtype)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    st = fa.fa_fwd_debug(q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(), lse.data_ptr(),
                         B, H, N, d, 0.125, 0, dtype, s, 1, 0.05)
    assert st == fa.FA_OK
    assert fa.fa_check_device_status(s) == fa.FA_ERR_TIMEOUT
    assert fa.fa_check_device_status(s) == fa.FA_OK          # cleared
    o2, lse2, _ = parity.run_gpu(q_bits, q_bits, q_bits, dtype, 0.125, False)
    rows = np.arange(N, dtype=np.int64)
    o_ref, lse_ref, spread = parity.oracle_rows(q_bits, q_bits, q_bits, dtype, 0.125, False, rows)
    parity.assert_within(parity.compare(o2.reshape(-1, d), lse2.reshape(-1), o_ref, lse_ref,
                                        spread, dtype), "after timeout")


def test_failed_launch_reports_fa_err_cuda_and_writes_nothing():
    """The launch step reporting failure (fa_fwd_debug fault_mode 2: the
    library returns as it would for a failed cudaLaunchKernel) comes back as
    FA_ERR_CUDA with nothing enqueued: O and LSE keep their canary values, the
    device status stays FA_OK and the next call is correct."""
    import torch
    import online_softmax_tiling_gb300 as fa
    B, H, N, d, dtype = 1, 2, 200, 128, synth.BF16
    q_bits = synth.tensor_bits(81, (B, H, N, d), dtype)
    q = parity.to_device(q_bits, dtype)
    o = torch.full_like(q, -1000.0)
    lse = torch.full((B, H, N), -1000.0, dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    for causal in (0, 1):
        st = fa.fa_fwd_debug(q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(),
                             lse.data_ptr(), B, H, N, d, 0.1, causal, dtype, s, 2, 2.0)
        assert st == fa.FA_ERR_CUDA
    assert fa.fa_check_device_status(s) == fa.FA_OK
    assert bool((o.float() == -1000.0).all()) and bool((lse == -1000.0).all())
    with pytest.raises(fa.FaError) as err:
        raise fa.FaError(fa.FA_ERR_CUDA)
    assert "FA_ERR_CUDA" in str(err.value)
    o2, lse2, _ = parity.run_gpu(q_bits, q_bits, q_bits, dtype, 0.1, True)
    rows = np.arange(B * H * N, dtype=np.int64)
    o_ref, lse_ref, spread = parity.oracle_rows(q_bits, q_bits, q_bits, dtype, 0.1, True, rows)
    parity.assert_within(parity.compare(o2.reshape(-1, d), lse2.reshape(-1), o_ref, lse_ref,
                                        spread, dtype), "after a failed launch")


def test_checked_wrapper_raises_on_a_timed_out_kernel():
    """attention_forward(check=True) turns a device-side FA_ERR_TIMEOUT into an
    exception instead of returning outputs that were never written."""
    import torch
    import online_softmax_tiling_gb300 as fa
    B, H, N, d, dtype = 1, 1, 256, 64, synth.FP16
    q = parity.to_device(synth.tensor_bits(91, (B, H, N, d), dtype), dtype)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert fa.fa_fwd_debug(q.data_ptr(), q.data_ptr(), q.data_ptr(), o.data_ptr(),
                           lse.data_ptr(), B, H, N, d, 0.125, 0, dtype, s, 1, 0.05) == fa.FA_OK
    with pytest.raises(fa.FaError) as err:
        fa._checked(s, "fa_fwd")
    assert err.value.status == fa.FA_ERR_TIMEOUT
    out, _ = fa.attention_forward(q, q, q, scale=0.125, check=True)   # status cleared, then OK
    assert torch.isfinite(out.float()).all()
