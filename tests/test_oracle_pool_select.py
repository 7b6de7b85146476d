"""Pins for the oracle's block pooling, block scores and hybrid block selection.

Closed forms for block means and scores; brute-force enumeration of all subsets
for the selection rule on small rows; invariants on larger rows.
"""
import itertools
import math

import numpy as np
import pytest

from oracle import prism_oracle as po
from audio_diffusion_dits_zone_b300 import synth


def test_block_mean_closed_forms():
    N, Hh, d, B = 10, 2, 3, 4      # blocks of 4, 4 and 2 tokens
    X = np.zeros((N, Hh, d))
    X[:, 0, 0] = np.arange(N)        # ramp: block means are the midpoints 1.5, 5.5, 8.5
    X[:, 1, :] = 7.0                 # constant
    m = po.block_mean(X, B)
    np.testing.assert_allclose(m[0, :, 0], [1.5, 5.5, 8.5])
    np.testing.assert_allclose(m[1], 7.0)
    assert po.block_lengths(N, B).tolist() == [4, 4, 2]


def test_scores_scale_and_bilinearity():
    d = 64
    e = np.eye(d)
    qbar = np.stack([e[:3]])           # [1, 3, d]
    kbar = np.stack([e[[0, 1, 5]]])
    S = po.block_scores(qbar, kbar)
    np.testing.assert_allclose(S[0], np.diag([1.0, 1.0, 0.0]) / math.sqrt(d))
    rng = np.random.default_rng(0)
    a, b, k = rng.normal(size=(3, 1, 4, d))
    np.testing.assert_allclose(po.block_scores(a + b, k),
                               po.block_scores(a, k) + po.block_scores(b, k))
    np.testing.assert_allclose(po.block_scores(a, k)[0], a[0] @ k[0].T / 8.0)


def test_pool_score_uses_block_order():
    rng = np.random.default_rng(5)
    N, Hh, d, B = 12, 1, 4, 4
    Q = rng.normal(size=(N, Hh, d))
    perm = np.arange(N)[::-1].copy()
    qbar, kbar, S = po.pool_score(Q, Q, perm, B)
    np.testing.assert_allclose(qbar[0, 0], Q[[11, 10, 9, 8], 0].mean(axis=0))
    np.testing.assert_allclose(S[0, 1, 2], qbar[0, 1] @ kbar[0, 2] / 2.0)


def brute_force_kept(s, sparsity, tau):
    """All subsets: top-k by (score desc, index asc) union the smallest-cardinality
    set whose softmax mass reaches tau (largest-mass one among those of that size,
    which is the top-m set)."""
    s = np.asarray(s, np.float64)
    nb = s.size
    p = np.exp(s - s.max())
    p /= p.sum()
    k = min(nb, max(1, math.ceil((1 - sparsity) * nb - 1e-9)))
    rank = sorted(range(nb), key=lambda j: (-s[j], j))
    top_k = set(rank[:k])
    best = None
    for size in range(1, nb + 1):
        for A in itertools.combinations(range(nb), size):
            if sum(p[list(A)]) >= tau:
                best = size
                break
        if best is not None:
            break
    top_m = set(rank[:best])
    return sorted(top_k | top_m), k, best


@pytest.mark.parametrize("seed", range(6))
def test_select_matches_brute_force(seed):
    rng = np.random.default_rng(seed)
    for _ in range(25):
        nb = int(rng.integers(2, 11))
        s = (rng.normal(size=nb) * rng.uniform(0.05, 4.0)).astype(np.float32)
        if rng.uniform() < 0.3:
            s = np.round(s * 2) / 2          # exact ties
        for sp in (0.0, 0.5, 0.75, 0.8, 0.93):
            for tau in (0.2, 0.5, 0.9):
                kept, k, m = po.select_row(s, sp, tau)
                bf, bk, bm = brute_force_kept(s, sp, tau)
                assert kept.tolist() == bf and k == bk and m == bm


def test_select_invariants_large_rows():
    S = synth.gen_scores(591, 64, seed=7)
    for row in S:
        for sp in (0.75, 0.8, 0.85, 0.93):
            kept, k, m = po.select_row(row, sp, 0.2)
            r = kept.size
            assert r == max(k, m) and r >= k
            order = po.descending_order(row.astype(np.float64))
            assert set(order[:k]) <= set(kept.tolist())
            p = np.exp(row - row.max())
            p /= p.sum()
            assert p[kept].sum() >= 0.2 - 1e-12
            if r > k:   # the CDF rule forced the extra blocks: one fewer misses tau
                assert p[order[: r - 1]].sum() < 0.2
            assert np.all(np.diff(kept) > 0)


def test_select_special_cases():
    # s = 0 keeps every block.
    kept, _, _ = po.select_row(np.arange(7, dtype=np.float32), 0.0, 0.2)
    assert kept.tolist() == list(range(7))
    # Uniform scores: p = 1/nb, m = ceil(tau nb); ties go to the lowest indices.
    nb = 32                       # p = 1/32 exactly: m = ceil(0.2 * 32) = 7, k = ceil(2.24) = 3
    kept, k, m = po.select_row(np.zeros(nb, np.float32), 0.93, 0.2)
    assert k == 3 and m == 7 and kept.tolist() == list(range(7))
    # k is exact when (1 - s) nb is an integer: 0.75 * ... -> (1 - 0.75) * 8 = 2
    assert po.keep_count_topk(8, 0.75) == 2
    assert po.keep_count_topk(591, 0.8) == 119
    assert po.keep_count_topk(1339, 0.85) == 201
    assert po.keep_count_topk(2363, 0.93) == 166
    assert po.keep_count_topk(10, 0.75) == 3
    # One dominant block: m = 1; top-k decides.
    s = np.full(20, -30.0, np.float32)
    s[13] = 0.0
    kept, k, m = po.select_row(s, 0.9, 0.2)
    assert m == 1 and k == 2 and kept.tolist() == [0, 13]


def test_select_decides_on_fp32_scores():
    # Two fp64 scores that round to the same fp32 value tie, and the smaller index wins.
    a = 1.0
    b = a + 1e-12
    kept, _, _ = po.select_row(np.array([a, b, -5.0, -5.0]), 0.75, 0.01)
    assert kept.tolist() == [0]
