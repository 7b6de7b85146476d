"""Comparison rules shared by the GPU parity tests.

Tolerances:
  * attention outputs and gradients, bf16 inputs with fp32 accumulation:
    max-abs <= 2e-2 and mean-abs <= 2e-3;
  * fp32 inputs (CUDA-core path): max-abs <= 2e-4 (fp32 accumulation over at most a
    few thousand terms of magnitude <= 1 has rounding error ~1e-5);
  * block indices bit-exact, except where the decision is a near-tie:
      - two scores within 1e-5 relative of each other (the stated tie rule), widened
        by twice the realised error of the library's fp32 scores on that row (two
        scores each off by at most e can swap order only when they are within 2e);
      - the cumulative softmax mass at the cut within MASS_TOL + 4e of the
        threshold.  The library sums exact fixed-point masses, so its only mass
        error is the single-precision exponential of each block (a few 1e-7
        relative) and the scores' own error e, which moves every mass by a factor
        within exp(+-2e).
    Every accepted row is classified (exact / score tie / mass band) so that the
    tests can bound how many rows pass only through a band.
"""
from __future__ import annotations

import numpy as np

U32 = 2.0 ** -24
# mass error of the selection kernel: expf is within a few ulp (~2.4e-7 relative) for
# every block, so prefix and total masses are each within that relative error; the
# fixed-point rounding adds at most 2^-41 of the largest block's mass per block
MASS_TOL = 1e-6


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


def classify_row(gpu_kept, s_ref, sparsity, tau, score_err=0.0):
    """How the library's kept set for the row s_ref is acceptable: "exact" (equal to the
    oracle's), "mass" (it takes a neighbouring cut whose oracle prefix mass lies within
    the mass band of tau), "score" (same length, differs only among near-tied scores),
    or None when it is not acceptable.

    s_ref is the oracle's score row; score_err the realised error of the library's
    scores on this row (max |library - oracle|).  The kept set must hold r blocks for
    an r the oracle allows, contain every block scoring clearly above the r-th score
    and none clearly below it.
    """
    from oracle import prism_oracle as po

    s = np.asarray(s_ref, np.float64)
    nb = s.size
    g = np.asarray(gpu_kept)
    if g.size and (np.any(np.diff(g) <= 0) or g[0] < 0 or g[-1] >= nb):
        return None
    ref, _, _ = po.select_row(s, sparsity, tau)
    if np.array_equal(g, ref):
        return "exact"
    order = po.descending_order(s)
    k = po.keep_count_topk(nb, sparsity)
    p = np.exp(s - s.max())
    p /= p.sum()
    cum = np.cumsum(p[order])
    mtol = MASS_TOL + 4.0 * score_err
    r0 = ref.size
    rs = {r0}
    for m in range(1, nb + 1):
        if abs(cum[m - 1] - tau) <= mtol:
            rs.update({max(k, m), max(k, min(m + 1, nb))})
    r = g.size
    if r not in rs:
        return None
    cut = s[order[r - 1]]
    tol = 1e-5 * np.maximum(np.abs(cut), np.abs(s)) + 2.0 * score_err
    forced_in = s > cut + tol
    forced_out = s < cut - tol
    inside = np.zeros(nb, bool)
    inside[g] = True
    if not (np.all(inside[forced_in]) and not np.any(inside[forced_out])):
        return None
    return "score" if r == r0 else "mass"


def check_row(gpu_kept, s_ref, sparsity, tau, score_err=0.0):
    """True if the library's kept set is an acceptable answer for the row s_ref."""
    return classify_row(gpu_kept, s_ref, sparsity, tau, score_err) is not None


def check_lists(counts, idx, s_ref, sparsity, tau, score_err=None):
    """Check every row; returns a dict of counts {rows, exact, score, mass} and the set of
    (h, i) rows whose list equals the oracle's; raises on a bad row.

    score_err: [Hh, nb] realised error of the library's scores per row (None = 0)."""
    Hh, nb = counts.shape
    stats = {"rows": Hh * nb, "exact": 0, "score": 0, "mass": 0}
    same = set()
    for h in range(Hh):
        for i in range(nb):
            g = idx[h, i, : counts[h, i]]
            e = 0.0 if score_err is None else float(score_err[h, i])
            how = classify_row(g, s_ref[h, i], sparsity, tau, e)
            assert how is not None, f"row (h={h}, i={i}): library kept {g.tolist()}"
            stats[how] += 1
            if how == "exact":
                same.add((h, i))
    return stats, same


def tie_budget(rows):
    """Most rows a workload may accept through a tie band: 1% of them, at least 2.
    A drift of the selection kernel shows up as many band rows, not a handful."""
    return max(2, rows // 100)


def record(name, entry):
    """Append one JSON line of parity statistics to $PRISM_PARITY_LOG, if it is set."""
    import json
    import os

    path = os.environ.get("PRISM_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps({"case": name, **entry}) + "\n")


def compare_perm_by_zone(gperm, operm, gzs, ozs, grid, zext):
    """Compare the permutation zone by zone for every zone whose chosen shape agrees.

    Each zone's tokens form one contiguous run of the block order, at an offset fixed by
    the sizes of the zones before it (independent of their shapes), so a zone whose
    shape differs on a near-tie leaves every other zone's run comparable.  Returns the
    number of zones compared; raises on the first run that differs."""
    from oracle import prism_oracle as po

    off = 0
    compared = 0
    for z, (t0, t1, h0, h1, w0, w1) in enumerate(po.zone_boxes(grid, zext)):
        n = (t1 - t0) * (h1 - h0) * (w1 - w0)
        if gzs[z] == ozs[z]:
            assert np.array_equal(gperm[off:off + n], operm[off:off + n]), f"zone {z}: permutation run differs"
            compared += 1
        off += n
    assert off == len(operm) == len(gperm)
    return compared
