"""The selection kernels' algorithm, restated in numpy, against a plain sort on CPU.

"Prism: dynamic sparse attention for 2K joint video-audio generation training",
section "Region-adapted block construction", paragraph 2 (hybrid selection: top
(1 - s) of the blocks and the shortest prefix whose softmax mass reaches the CDF
threshold).  The kernels never sort a row: they drop the scores into equal-width
buckets, find the bucket where both conditions are first met scanning from the
top, and rank only that bucket's blocks exactly.  This test pins the claim that the
result is the sorted-prefix answer exactly, for any monotone bucketing, including
ties (equal scores go to the smaller index) and flat rows; both sides use the same
fixed-point masses q = round(exp(s - max) * 2^40), as the kernels do, so the
comparison is exact.
"""
import math

import numpy as np
import pytest

from audio_diffusion_dits_zone_b300 import synth

SCALE = float(2 ** 40)


def masses(s):
    s = np.asarray(s, np.float32)
    return np.rint(np.exp((s - s.max()).astype(np.float32)).astype(np.float64) * SCALE).astype(np.uint64)


def target_of(q, tau):
    z = int(q.sum(dtype=np.uint64))
    t = math.ceil(tau * float(z))
    return min(z, t)


def k_of(nb, sparsity):
    return int(min(nb, max(1, math.ceil((1.0 - sparsity) * nb - 1e-9))))


def sorted_prefix(s, sparsity, tau):
    """The definition: descending score (smaller index first on ties); the shortest
    prefix with at least k blocks and at least the target mass."""
    s = np.asarray(s, np.float32)
    nb = s.size
    q = masses(s)
    order = np.lexsort((np.arange(nb), -s.astype(np.float64)))
    k, target = k_of(nb, sparsity), target_of(q, tau)
    run = 0
    for r, j in enumerate(order, start=1):
        run += int(q[j])
        if r >= k and run >= target:
            return np.sort(order[:r])
    return np.sort(order)


def bucketed(s, sparsity, tau, bins=256):
    """The kernels' steps: buckets, crossing bucket, exact ranking inside it."""
    s = np.asarray(s, np.float32)
    nb = s.size
    q = masses(s)
    k, target = k_of(nb, sparsity), target_of(q, tau)
    mn, mx = s.min(), s.max()
    rng = np.float32(mx - mn)
    scale = np.float32(bins) / rng if rng > 0 else np.float32(0)
    b = np.clip(np.trunc((s - mn) * scale).astype(np.int64), 0, bins - 1)  # monotone in s
    cnt = np.bincount(b, minlength=bins)
    mass = np.zeros(bins, dtype=object)
    for j in range(nb):
        mass[b[j]] += int(q[j])
    c_run, m_run, bstar = 0, 0, None
    for x in range(bins - 1, -1, -1):
        if cnt[x] > 0 and c_run + cnt[x] >= k and m_run + mass[x] >= target:
            bstar = x
            break
        c_run += int(cnt[x])
        m_run += mass[x]
    assert bstar is not None  # every block counted: both conditions hold
    kept = b > bstar
    cand = np.nonzero(b == bstar)[0]  # index order
    keys = s[cand].astype(np.float64)
    if keys.min() == keys.max():
        qv = int(q[cand[0]])
        tk = max(0, k - c_run)
        tm = 0 if m_run >= target else (min(len(cand), -(-(target - m_run) // qv)) if qv > 0 else len(cand))
        best = min(len(cand), max(tk, tm))
        kept[cand[:best]] = True
    else:
        ranks, take = [], len(cand)
        for c, i in enumerate(cand):
            before = [d for d in range(len(cand)) if keys[d] > keys[c] or (keys[d] == keys[c] and cand[d] < i)]
            rank = len(before)
            pre = sum(int(q[cand[d]]) for d in before)
            ranks.append(rank)
            if c_run + rank + 1 >= k and m_run + pre + int(q[i]) >= target:
                take = min(take, rank + 1)
        for c, i in enumerate(cand):
            if ranks[c] < take:
                kept[i] = True
    return np.nonzero(kept)[0]


@pytest.mark.parametrize("bins", [256, 16, 1])
def test_buckets_give_the_sorted_prefix(bins):
    cases = 0
    for nb, sp, ties in ((10, 0.75, False), (64, 0.8, True), (200, 0.5, False), (300, 0.93, True), (591, 0.8, False)):
        rows = synth.gen_scores(nb, 12, seed=nb + bins, ties=ties)
        for r in rows:
            for tau in (0.0, 0.2, 0.9):
                assert np.array_equal(bucketed(r, sp, tau, bins), sorted_prefix(r, sp, tau)), (nb, sp, tau, bins)
                cases += 1
    assert cases == 5 * 12 * 3


def test_flat_rows_and_one_outlier():
    nb = 100
    for sp in (0.75, 0.93):
        flat = np.full(nb, 2.5, np.float32)
        assert np.array_equal(bucketed(flat, sp, 0.2), sorted_prefix(flat, sp, 0.2))
        assert bucketed(flat, sp, 0.2).tolist() == list(range(max(k_of(nb, sp), 20)))
        spike = flat.copy()
        spike[37] = 9.0  # one block holds almost all the mass: the CDF cut is one block
        got = bucketed(spike, sp, 0.2)
        assert np.array_equal(got, sorted_prefix(spike, sp, 0.2)) and 37 in got
