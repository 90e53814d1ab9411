"""Pins for the CPU oracle: what the pages and the mathematics fix.

Each check ties the oracle to something other than itself: the worked example
printed in "用 CuTe 读懂 FlashAttention：一次 forward 的完整流程" (Fig. 5-12), the
causal variant of Fig. 11, closed forms, invariants of softmax attention, a
library softmax / log-sum-exp, and brute force in 50-digit arithmetic.
"""
import math

import numpy as np
import pytest

import oracle
from tests.golden import fixtures

EXACT = 1e-14


def _ex():
    return fixtures.load("worked_example.txt")


def test_worked_example_plain_definition():
    ex = _ex()
    o, lse = oracle.attention(ex["Q"], ex["K"], ex["V"], ex["scale"])
    np.testing.assert_allclose(o, ex["O"], rtol=0, atol=EXACT)
    np.testing.assert_allclose(lse, ex["LSE"], rtol=0, atol=EXACT)


def test_worked_example_recurrence_intermediates():
    ex = _ex()
    o, lse, tr = oracle.blocked_head(ex["Q"], ex["K"], ex["V"], ex["scale"], False,
                                     int(ex["block_n"]), trace=True)
    # key block 0 (Fig. 6, Fig. 8, l0 = 3/2, m = 1); no rescale on the first block
    np.testing.assert_allclose(tr["m"][0], ex["m0"], atol=EXACT)
    np.testing.assert_allclose(tr["e"][0], ex["E0"], atol=EXACT)
    np.testing.assert_allclose(tr["l"][0], ex["l0"], atol=EXACT)
    np.testing.assert_allclose(tr["u"][0], ex["U0"], atol=EXACT)
    assert np.all(np.isnan(tr["alpha"][0]))
    # key block 1 (alpha = 1/2, Fig. 7, l1, Fig. 9, Fig. 10)
    np.testing.assert_allclose(tr["m"][1], ex["m1"], atol=EXACT)
    np.testing.assert_allclose(tr["alpha"][1], ex["alpha1"], atol=EXACT)
    np.testing.assert_allclose(tr["e"][1], ex["E1"], atol=EXACT)
    np.testing.assert_allclose(tr["l"][1], ex["l1"], atol=EXACT)
    np.testing.assert_allclose(tr["u"][1], ex["U1"], atol=EXACT)
    du = tr["u"][1] - tr["alpha"][1][:, None] * tr["u"][0]
    np.testing.assert_allclose(du, ex["dU1"], atol=EXACT)
    # raw scores of Fig. 5 recovered from the weights: e = 2^(x - m) when s = ln 2
    s_rec = np.concatenate([np.log2(tr["e"][t]) + tr["m"][t][:, None] for t in range(2)],
                           axis=1)
    np.testing.assert_allclose(s_rec, ex["S"], atol=1e-12)
    np.testing.assert_allclose(o, ex["O"], atol=EXACT)
    np.testing.assert_allclose(lse, ex["LSE"], atol=EXACT)


def test_worked_example_causal():
    ex = _ex()
    cz = fixtures.load("worked_example_causal.txt")
    o, lse = oracle.attention(ex["Q"], ex["K"], ex["V"], cz["scale"], causal=True)
    np.testing.assert_allclose(o, cz["O"], atol=EXACT)
    np.testing.assert_allclose(lse, cz["LSE"], atol=EXACT)
    ob, lseb, tr = oracle.blocked_head(ex["Q"], ex["K"], ex["V"], cz["scale"], True,
                                       int(cz["block_n"]), trace=True)
    np.testing.assert_allclose(ob, cz["O"], atol=EXACT)
    np.testing.assert_allclose(lseb, cz["LSE"], atol=EXACT)
    # Fig. 11: masked positions carry no weight; the future block is skipped
    masked = np.isinf(cz["S_causal"][:, :2])
    assert np.all(tr["e"][0][masked] == 0.0)
    k = int(cz["skipped_block"])
    assert np.all(tr["e"][k] == 0.0) and np.all(np.isnan(tr["alpha"][k]))
    np.testing.assert_array_equal(tr["l"][k], tr["l"][0])


def _rand_case(rng, n, d, scale_hi=1.5):
    q = rng.standard_normal((n, d))
    k = rng.standard_normal((n, d))
    v = rng.standard_normal((n, d))
    s = float(rng.uniform(0.05, scale_hi))
    return q, k, v, s


@pytest.mark.parametrize("causal", [False, True])
def test_recurrence_equals_plain_definition_for_every_block_size(causal):
    rng = np.random.default_rng(11)
    for n in range(1, 10):
        for d in (1, 2, 3, 5):
            q, k, v, s = _rand_case(rng, n, d)
            o_ref, lse_ref = oracle.attention(q, k, v, s, causal)
            for bn in range(1, n + 2):
                o, lse = oracle.blocked_head(q, k, v, s, causal, bn)
                np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
                np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_probabilities_match_library_softmax_and_sum_to_one(causal):
    from scipy.special import logsumexp, softmax
    rng = np.random.default_rng(5)
    n = 7
    q, k, _, s = _rand_case(rng, n, n)
    v = np.eye(n)                       # O row i is then the probability row P_i
    p, lse = oracle.attention(q, k, v, s, causal)
    scores = s * (q @ k.T)
    for i in range(n):
        nv = i + 1 if causal else n
        np.testing.assert_allclose(p[i, :nv], softmax(scores[i, :nv]), atol=1e-14)
        np.testing.assert_allclose(p[i, nv:], 0.0, atol=0)
        assert abs(p[i].sum() - 1.0) < 1e-14
        assert abs(lse[i] - logsumexp(scores[i, :nv])) < 1e-13


def test_key_permutation_invariance_noncausal():
    rng = np.random.default_rng(7)
    q, k, v, s = _rand_case(rng, 9, 4)
    o, lse = oracle.attention(q, k, v, s)
    perm = rng.permutation(9)
    o2, lse2 = oracle.attention(q, k[perm], v[perm], s)
    np.testing.assert_allclose(o2, o, atol=1e-14)
    np.testing.assert_allclose(lse2, lse, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_convex_combination_and_lse_bounds(causal):
    rng = np.random.default_rng(3)
    q, k, v, s = _rand_case(rng, 12, 6)
    o, lse = oracle.attention(q, k, v, s, causal)
    x = q @ k.T
    for i in range(12):
        nv = i + 1 if causal else 12
        lo, hi = v[:nv].min(axis=0), v[:nv].max(axis=0)
        assert np.all(o[i] >= lo - 1e-14) and np.all(o[i] <= hi + 1e-14)
        m = x[i, :nv].max()
        assert s * m - 1e-14 <= lse[i] <= s * m + math.log(nv) + 1e-14


def test_single_key_gives_value_row():
    rng = np.random.default_rng(9)
    q, k, v, s = _rand_case(rng, 1, 8)
    o, lse = oracle.attention(q, k, v, s)
    np.testing.assert_array_equal(o, v)
    assert abs(lse[0] - s * float(q[0] @ k[0])) < 1e-14


@pytest.mark.parametrize("causal", [False, True])
def test_zero_queries_give_uniform_weights(causal):
    rng = np.random.default_rng(13)
    _, k, v, s = _rand_case(rng, 10, 3)
    q = np.zeros_like(k)
    o, lse = oracle.attention(q, k, v, s, causal)
    for i in range(10):
        nv = i + 1 if causal else 10
        np.testing.assert_allclose(o[i], v[:nv].mean(axis=0), atol=1e-14)
        assert abs(lse[i] - math.log(nv)) < 1e-14


def test_constant_values_give_constant_output():
    rng = np.random.default_rng(17)
    q, k, _, s = _rand_case(rng, 8, 5)
    c = rng.standard_normal(5)
    v = np.tile(c, (8, 1))
    for causal in (False, True):
        o, _ = oracle.attention(q, k, v, s, causal)
        np.testing.assert_allclose(o, np.tile(c, (8, 1)), atol=1e-14)


def test_dominant_key_selects_its_value():
    rng = np.random.default_rng(19)
    q, k, v, _ = _rand_case(rng, 6, 4)
    k[4] = 40.0 * q[2] / np.linalg.norm(q[2]) ** 2      # q2 . k4 = 40, others O(1)
    o, _ = oracle.attention(q, k, v, 1.0)
    np.testing.assert_allclose(o[2], v[4], atol=1e-12)


def test_brute_force_fifty_digits():
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 50
    rng = np.random.default_rng(23)
    for n, d, causal in [(1, 1, False), (3, 2, True), (5, 4, False), (8, 3, True), (7, 4, False)]:
        q, k, v, s = _rand_case(rng, n, d, scale_hi=3.0)
        o, lse = oracle.attention(q, k, v, s, causal)
        for i in range(n):
            nv = i + 1 if causal else n
            xs = [mpmath.fsum(mpmath.mpf(q[i, c]) * mpmath.mpf(k[j, c]) for c in range(d))
                  for j in range(nv)]
            ws = [mpmath.exp(mpmath.mpf(s) * x) for x in xs]     # no max subtraction
            tot = mpmath.fsum(ws)
            for c in range(d):
                ref = mpmath.fsum(w * mpmath.mpf(v[j, c]) for j, w in enumerate(ws)) / tot
                assert abs(float(ref) - o[i, c]) < 1e-13
            assert abs(float(mpmath.log(tot)) - lse[i]) < 1e-13


def test_decode16_exhaustive_against_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f16 = oracle.decode16(bits, oracle.FP16)
    ref16 = bits.view(np.float16).astype(np.float64)
    same = (f16 == ref16) | (np.isnan(f16) & np.isnan(ref16))
    assert same.all()
    b16 = oracle.decode16(bits, oracle.BF16)
    with np.errstate(invalid="ignore"):
        refb = (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    same = (b16 == refb) | (np.isnan(b16) & np.isnan(refb))
    assert same.all()


@pytest.mark.parametrize("dtype", [oracle.FP16, oracle.BF16])
@pytest.mark.parametrize("causal", [False, True])
def test_rows16_matches_widened_definition(dtype, causal):
    from online_softmax_tiling_gb300 import synth
    B, H, N, d = 1, 3, 37, 16
    q = synth.tensor_bits(91, (B, H, N, d), dtype)
    k = synth.tensor_bits(92, (B, H, N, d), dtype)
    v = synth.tensor_bits(93, (B, H, N, d), dtype)
    s = 0.25
    o_all, lse_all = oracle.attention(oracle.decode16(q, dtype), oracle.decode16(k, dtype),
                                      oracle.decode16(v, dtype), s, causal)
    rows = np.array([0, 5, N - 1, N, 2 * N + 17, 3 * N - 1, 40], dtype=np.int64)
    o, lse = oracle.attention_rows16(q, k, v, dtype, s, causal, rows, nthreads=3)
    np.testing.assert_array_equal(o, o_all.reshape(-1, d)[rows])
    np.testing.assert_array_equal(lse, lse_all.reshape(-1)[rows])


def test_spread_matches_brute_force_and_closed_form():
    from online_softmax_tiling_gb300 import synth
    dtype, N, d, s = oracle.BF16, 23, 8, 0.3
    q = synth.tensor_bits(31, (1, 2, N, d), dtype)
    k = synth.tensor_bits(32, (1, 2, N, d), dtype)
    v = synth.tensor_bits(33, (1, 2, N, d), dtype)
    Q, K, V = (oracle.decode16(t, dtype)[0] for t in (q, k, v))
    rows = np.arange(2 * N, dtype=np.int64)
    for causal in (False, True):
        o, _, spread = oracle.attention_rows16(q, k, v, dtype, s, causal, rows, with_spread=True)
        for r in rows:
            h, i = divmod(int(r), N)
            nv = i + 1 if causal else N
            x = s * (Q[h, i] @ K[h, :nv].T)
            p = np.exp(x - x.max())
            p /= p.sum()
            want = (p[:, None] * np.abs(V[h, :nv] - o[r][None, :])).sum(0)
            np.testing.assert_allclose(spread[r], want, rtol=1e-12, atol=1e-15)
    # two keys with equal scores: weights 1/2 each, spread = |v0 - v1| / 2
    qq = np.zeros((1, 1, 2, 2), np.uint16)
    vv = synth.round_to_bits(np.array([[[[1.0, -2.0], [3.0, 0.5]]]]), oracle.FP16)
    _, _, sp = oracle.attention_rows16(qq, qq, vv, oracle.FP16, 1.0, False, [0, 1],
                                       with_spread=True)
    np.testing.assert_allclose(sp, [[1.0, 1.25], [1.0, 1.25]], atol=1e-15)


def test_worked_example_bottom_right():
    ex = _ex()
    br = fixtures.load("worked_example_bottom_right.txt")
    o, lse = oracle.attention(ex["Q"], ex["K"], ex["V"], br["scale"], oracle.BOTTOM_RIGHT)
    np.testing.assert_allclose(o, br["O"], atol=EXACT)
    np.testing.assert_allclose(lse, br["LSE"], atol=EXACT)
    ob, lb = oracle.blocked_head(ex["Q"], ex["K"], ex["V"], br["scale"], oracle.BOTTOM_RIGHT, 2)
    np.testing.assert_allclose(ob, br["O"], atol=EXACT)
    np.testing.assert_allclose(lb, br["LSE"], atol=EXACT)


def test_bottom_right_special_cases():
    rng = np.random.default_rng(29)
    # equal lengths: bottom-right is top-left
    q, k, v, s = _rand_case(rng, 9, 4)
    a = oracle.attention(q, k, v, s, oracle.TOP_LEFT)
    b = oracle.attention(q, k, v, s, oracle.BOTTOM_RIGHT)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])
    # one query (decoding): it sees every key
    q1 = rng.standard_normal((1, 4))
    a = oracle.attention(q1, k, v, s, oracle.NO_MASK)
    b = oracle.attention(q1, k, v, s, oracle.BOTTOM_RIGHT)
    np.testing.assert_array_equal(a[0], b[0])
    # more queries than keys: the first Nq - Nk rows see nothing, the next sees key 0
    q7 = rng.standard_normal((7, 4))
    k3, v3 = k[:3], v[:3]
    o, lse = oracle.attention(q7, k3, v3, s, oracle.BOTTOM_RIGHT)
    np.testing.assert_array_equal(o[:4], 0.0)
    assert np.all(np.isneginf(lse[:4]))
    np.testing.assert_allclose(o[4], v3[0], atol=1e-15)
    assert abs(lse[4] - s * float(q7[4] @ k3[0])) < 1e-14


@pytest.mark.parametrize("nq,nk", [(3, 8), (8, 3), (5, 5), (1, 9), (9, 1)])
def test_recurrence_equals_plain_definition_unequal_lengths(nq, nk):
    rng = np.random.default_rng(100 + nq * 10 + nk)
    q = rng.standard_normal((nq, 3))
    k = rng.standard_normal((nk, 3))
    v = rng.standard_normal((nk, 3))
    for mask in (oracle.NO_MASK, oracle.TOP_LEFT, oracle.BOTTOM_RIGHT):
        o_ref, lse_ref = oracle.attention(q, k, v, 0.6, mask)
        for bn in range(1, nk + 2):
            o, lse = oracle.blocked_head(q, k, v, 0.6, mask, bn)
            np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
            np.testing.assert_array_equal(np.isneginf(lse), np.isneginf(lse_ref))
            fin = np.isfinite(lse_ref)
            np.testing.assert_allclose(lse[fin], lse_ref[fin], rtol=0, atol=1e-12)


def test_brute_force_unequal_lengths_bottom_right():
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 50
    rng = np.random.default_rng(37)
    for nq, nk in [(3, 7), (6, 4), (1, 5)]:
        q = rng.standard_normal((nq, 3))
        k = rng.standard_normal((nk, 3))
        v = rng.standard_normal((nk, 3))
        o, lse = oracle.attention(q, k, v, 0.9, oracle.BOTTOM_RIGHT)
        for i in range(nq):
            nv = min(nk, max(0, i + 1 + nk - nq))
            if nv == 0:
                assert np.all(o[i] == 0) and np.isneginf(lse[i])
                continue
            ws = [mpmath.exp(mpmath.mpf(0.9) * mpmath.fsum(mpmath.mpf(q[i, c]) * mpmath.mpf(k[j, c])
                                                         for c in range(3))) for j in range(nv)]
            tot = mpmath.fsum(ws)
            for c in range(3):
                ref = mpmath.fsum(w * mpmath.mpf(v[j, c]) for j, w in enumerate(ws)) / tot
                assert abs(float(ref) - o[i, c]) < 1e-13
            assert abs(float(mpmath.log(tot)) - lse[i]) < 1e-13


def test_rows16_unequal_lengths_match_widened_definition():
    from online_softmax_tiling_gb300 import synth
    dtype = oracle.BF16
    q = synth.tensor_bits(301, (1, 2, 13, 8), dtype)
    k = synth.tensor_bits(302, (1, 2, 29, 8), dtype)
    v = synth.tensor_bits(303, (1, 2, 29, 8), dtype)
    for mask in (oracle.NO_MASK, oracle.TOP_LEFT, oracle.BOTTOM_RIGHT):
        o_all, lse_all = oracle.attention(oracle.decode16(q, dtype), oracle.decode16(k, dtype),
                                          oracle.decode16(v, dtype), 0.3, mask)
        rows = np.arange(26, dtype=np.int64)
        o, lse = oracle.attention_rows16(q, k, v, dtype, 0.3, mask, rows)
        np.testing.assert_array_equal(o, o_all.reshape(-1, 8))
        np.testing.assert_array_equal(lse, lse_all.reshape(-1))
