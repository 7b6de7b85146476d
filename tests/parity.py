"""Comparison rules shared by the GPU parity tests.

Tolerances:
  * attention outputs and gradients, bf16 inputs with fp32 accumulation:
    max-abs <= 2e-2 and mean-abs <= 2e-3;
  * fp32 inputs (CUDA-core path): max-abs <= 2e-4 (fp32 accumulation over at most a
    few thousand terms of magnitude <= 1 has rounding error ~1e-5);
  * block indices bit-exact, except where the decision is a near-tie:
      - two scores within 1e-5 relative of each other, widened by the worst-case
        error of the library's fp32 score (below) when its scores are its own;
      - the cumulative softmax mass at the cut within nb * 2^-24 of the threshold
        (the worst-case relative error of a length-nb fp32 sum).
"""
from __future__ import annotations

import numpy as np

U32 = 2.0 ** -24


def attn_close(got, ref, max_abs=2e-2, mean_abs=2e-3, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    err = np.abs(got - ref)
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    mx, mn = float(err.max()), float(err.mean())
    assert mx <= max_abs and mn <= mean_abs, f"{what}: max-abs {mx:.3e} (<= {max_abs}), mean-abs {mn:.3e} (<= {mean_abs})"
    return mx, mn


def score_error_bound(qbar, kbar, d):
    """Worst-case |fp32 score - exact score| per (h, i) row, from the sizes of the block
    means: each mean of <= 128 values and the d-term dot product accumulate in fp32."""
    qn = np.linalg.norm(qbar, axis=-1)           # [Hh, nb]
    kn = np.linalg.norm(kbar, axis=-1).max(-1)   # [Hh]
    return 3.0 * (128 + d) * U32 * qn * kn[:, None] / np.sqrt(d)


def check_row(gpu_kept, s_ref, sparsity, tau, score_tol=0.0):
    """True if the library's kept set is an acceptable answer for the row s_ref.

    s_ref is the oracle's score row (fp64 or the fp32 input).  The kept set must hold
    r blocks for an r the oracle allows (r = max(k, m), or the neighbouring m when
    the mass at the cut is within the fp32 summation bound of tau), contain every
    block scoring clearly above the r-th score and none clearly below it.
    """
    from oracle import prism_oracle as po

    s = np.asarray(s_ref, np.float64)
    nb = s.size
    g = np.asarray(gpu_kept)
    if g.size and (np.any(np.diff(g) <= 0) or g[0] < 0 or g[-1] >= nb):
        return False
    order = po.descending_order(s)
    k = po.keep_count_topk(nb, sparsity)
    p = np.exp(s - s.max())
    p /= p.sum()
    cum = np.cumsum(p[order])
    mtol = nb * U32 * 4 + 1e-9
    ms = {int(np.argmax(cum >= tau)) + 1 if (cum >= tau).any() else nb}
    for m in range(1, nb + 1):
        if abs(cum[m - 1] - tau) <= mtol:
            ms.update({m, m + 1})
    rs = {max(k, min(m, nb)) for m in ms}
    r = g.size
    if r not in rs:
        return False
    cut = s[order[r - 1]]
    tol = 1e-5 * np.maximum(np.abs(cut), np.abs(s)) + 2 * score_tol
    forced_in = s > cut + tol
    forced_out = s < cut - tol
    inside = np.zeros(nb, bool)
    inside[g] = True
    return bool(np.all(inside[forced_in]) and not np.any(inside[forced_out]))


def check_lists(counts, idx, s_ref, sparsity, tau, score_tol=None):
    """Check every row; returns (n_rows, n_exact, n_tie_accepted); raises on a bad row."""
    from oracle import prism_oracle as po

    Hh, nb = counts.shape
    exact = tie = 0
    for h in range(Hh):
        for i in range(nb):
            g = idx[h, i, : counts[h, i]]
            ref, _, _ = po.select_row(s_ref[h, i], sparsity, tau)
            if np.array_equal(g, ref):
                exact += 1
                continue
            st = 0.0 if score_tol is None else float(score_tol[h, i])
            assert check_row(g, s_ref[h, i], sparsity, tau, st), \
                f"row (h={h}, i={i}): library kept {g.tolist()} vs oracle {ref.tolist()}"
            tie += 1
    return Hh * nb, exact, tie
