"""The split-KV merge's arithmetic ("CUDA 算子工程" 14.7.1) on the CPU: attention
over contiguous key ranges, each normalised by its own weight sum and
summarised by its log-sum-exp, recombined with weights e^{LSE_s - max}
gives the attention over all keys, and LSE = ln sum_s e^{LSE_s}.  The ranges
are split as the kernel splits a query block's visible key tiles, with the
causal mask and with ranges that are empty for some rows.  The recombined
result is compared with the oracle on the whole problem.  This pins the
reading the merge kernel implements, not the kernel itself, which the GPU
split-KV tests compare with the oracle."""
import numpy as np
import pytest

import oracle


def _range_partials(q, k, v, scale, causal, lo, hi):
    """O and LSE of every query row over keys [lo, hi) (plain float64; a row
    with no visible key in the range gets O = 0, LSE = -inf)."""
    Nq = q.shape[0]
    x = (q @ k[lo:hi].T) * scale
    if causal:
        keys = np.arange(lo, hi)[None, :]
        x = np.where(keys <= np.arange(Nq)[:, None], x, -np.inf)
    m = x.max(axis=1, initial=-np.inf)
    live = np.isfinite(m)
    e = np.exp(x - np.where(live, m, 0.0)[:, None])
    ell = e.sum(axis=1)
    o = np.zeros((Nq, v.shape[1]))
    o[live] = (e[live] @ v[lo:hi]) / ell[live, None]
    lse = np.full(Nq, -np.inf)
    lse[live] = m[live] + np.log(ell[live])
    return o, lse


def _merge(parts):
    """LSE-weighted recombination of (O_s, LSE_s) pairs, row by row."""
    lses = np.stack([l for _, l in parts])          # [S, Nq]
    mx = lses.max(axis=0)
    w = np.where(np.isfinite(lses), np.exp(lses - np.where(np.isfinite(mx), mx, 0.0)), 0.0)
    wsum = w.sum(axis=0)
    o = sum(w[s][:, None] * parts[s][0] for s in range(len(parts)))
    o = np.where(wsum[:, None] > 0, o / np.where(wsum > 0, wsum, 1.0)[:, None], 0.0)
    lse = np.where(wsum > 0, np.where(np.isfinite(mx), mx, 0.0) + np.log(np.where(wsum > 0, wsum, 1.0)),
                   -np.inf)
    return o, lse


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("S", [2, 3, 5, 32])
def test_ranges_recombine_to_the_whole(causal, S):
    rng = np.random.default_rng(100 + 7 * S + int(causal))
    Nq = Nk = 300
    d = 16
    q, k, v = (rng.standard_normal((n, d)) for n in (Nq, Nk, Nk))
    scale = 0.25
    # contiguous ranges of 128-key tiles, as the kernel cuts the visible
    # tiles of a block; with 32 ranges most are empty
    tiles = -(-Nk // 128)
    chunk = -(-tiles // S)
    bounds = [(min(s * chunk * 128, Nk), min((s + 1) * chunk * 128, Nk)) for s in range(S)]
    parts = [_range_partials(q, k, v, scale, causal, lo, hi) for lo, hi in bounds]
    o, lse = _merge(parts)
    o_ref, lse_ref = oracle.attention(q[None], k[None], v[None], scale, causal)
    np.testing.assert_allclose(o, o_ref[0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref[0], rtol=0, atol=1e-12)


def test_a_dropped_range_is_caught():
    """The comparison above is sensitive: merging all ranges but one differs."""
    rng = np.random.default_rng(9)
    q, k, v = (rng.standard_normal((256, 16)) for _ in range(3))
    bounds = [(0, 128), (128, 256)]
    parts = [_range_partials(q, k, v, 0.25, False, lo, hi) for lo, hi in bounds]
    o, _ = _merge(parts[:1])
    o_ref, _ = oracle.attention(q[None], k[None], v[None], 0.25, False)
    assert np.abs(o - o_ref[0]).max() > 1e-3
