"""CPU oracle for Prism-style dynamic block-sparse attention (fp64, numpy).

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or run
this module: only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` do.  It shares no code with the CUDA library: no kernels,
headers, helpers, tables or constants.  Its inputs come from the seeded input
module (``audio_diffusion_dits_zone_b300.synth``) or from the tests.

Source.  "Prism: dynamic sparse attention for 2K joint video-audio generation
training" (trawling.dev/post/2299, a summary of the Prism project page), section
"Region-adapted block construction":
  * paragraph 1 -- tokens are split into spatio-temporal macro-zones; in every
    zone the channel-wise variance of the video features and the feature norm of
    the audio-to-video cross-attention are measured; the first says along which
    axis and how fast the video changes, the second how strongly audio drives
    the region; both set the zone's block shape, dividing more finely along
    axes of fast change or strong audio-video coupling, so that block-level
    features are semantically tight;
  * paragraph 2 -- blocks are chosen by a hybrid strategy that makes the
    sparsity of every query dynamic; Prism Block Sparse Attention (BSA) runs on
    the chosen blocks; settings list BSA sparsity 0.75 / 0.80 / 0.85 / 0.93 and
    a CDF threshold of 0.20 for the hybrid selection.

The page gives no formulas.  Where it is silent this oracle takes the plainest
reading the text supports; each reading is stated where it is used:
  R1 zones tile the grid from the origin, the last zone on an axis is clipped,
     zones are numbered in raster order of (zone_t, zone_h, zone_w);
  R2 "channel-wise variance along an axis" = the population variance of each
     channel along every line of the zone parallel to that axis, averaged over
     the zone's lines and over channels; the video feature is V (all heads);
  R3 A2V coupling along an axis = the same line variance of the A2V norm field;
     its weight in a zone is the zone's mean A2V norm over the largest zone mean;
  R4 per-axis score S_a = v_a / sum_b v_b + w * u_a / sum_b u_b (0/0 := 0); the
     shape (e_t, e_h, e_w) of least cost sum_a S_a log2(e_a) wins, lowest index
     on ties, so a larger score gives a smaller extent along that axis;
  R5 block order: zones in raster order; inside a zone, tiles of the chosen
     shape in tile-raster order, clipped at the zone edge; inside a tile, tokens
     in raster order; blocks are consecutive B-token chunks of that sequence
     (only the last block can be short);
  R6 block features are block means of Q and K (true length for the short
     block); block score = qbar . kbar / sqrt(d);
  R7 hybrid selection keeps the union of the top ceil((1 - s) nb) blocks and the
     smallest prefix of the descending-score order whose softmax mass reaches the
     CDF threshold; both are prefixes of one order, so the union is the longer
     prefix; ties in score go to the smaller block index; no block is forced;
  R8 attention is plain softmax attention of each query token over all tokens of
     its query block's kept blocks, scale 1/sqrt(d), no causal mask; backward
     treats the kept lists as constants;
  R9 the A2V field is the feature norm of the audio-to-video cross-attention: each
     video token's query attends (softmax, scale 1/sqrt(d), per head) to every audio
     token; the field at the token is the L2 norm of its whole output feature, all
     heads' channels together.

Decisions that floating point makes (which shape, which block) are taken on the
values in the precision the library stores them in: scores are rounded to fp32
(the scores buffer is fp32) and zone costs are compared in fp32.
"""
from __future__ import annotations

import math

import numpy as np

AXES = 3  # t, h, w


# ----------------------------------------------------------------------------- zones
def zone_boxes(grid, zext):
    """Macro-zones as half-open boxes (t0, t1, h0, h1, w0, w1), raster order (R1)."""
    T, H, W = grid
    zt, zh, zw = zext
    boxes = []
    for t0 in range(0, T, zt):
        for h0 in range(0, H, zh):
            for w0 in range(0, W, zw):
                boxes.append((t0, min(t0 + zt, T), h0, min(h0 + zh, H), w0, min(w0 + zw, W)))
    return boxes


def line_variance_sum(X: np.ndarray, axis: int) -> np.ndarray:
    """Sum over channels of the mean over lines of the population variance along ``axis``.

    X is one zone, shape [Lt, Lh, Lw, C].  A line along axis a is the set of
    tokens that share the other two coordinates (R2).  A length-1 axis has no
    variation, so its value is 0.
    """
    if X.shape[axis] == 1:
        return 0.0
    var = X.var(axis=axis)  # population variance (ddof = 0) of every line and channel
    return float(var.mean(axis=(0, 1)).sum())


def zone_video_variation(feature_chunks, grid, zext) -> np.ndarray:
    """v[Z, 3]: per-zone, per-axis channel-wise variance of the video feature (R2).

    ``feature_chunks`` yields arrays [N, c] in raster token order whose channels
    together make up the feature (e.g. one head of V at a time); the result is
    averaged over all channels.
    """
    T, H, W = grid
    boxes = zone_boxes(grid, zext)
    acc = np.zeros((len(boxes), AXES), dtype=np.float64)
    C = 0
    for F in feature_chunks:
        F4 = np.asarray(F, dtype=np.float64).reshape(T, H, W, -1)
        C += F4.shape[-1]
        for z, (t0, t1, h0, h1, w0, w1) in enumerate(boxes):
            X = F4[t0:t1, h0:h1, w0:w1, :]
            for a in range(AXES):
                acc[z, a] += line_variance_sum(X, a)
    return acc / C


def zone_a2v_coupling(a2v, grid, zext):
    """(u[Z, 3], abar[Z]): per-axis line variance of the A2V field and zone mean (R3)."""
    T, H, W = grid
    A = np.asarray(a2v, dtype=np.float64).reshape(T, H, W, 1)
    boxes = zone_boxes(grid, zext)
    u = np.zeros((len(boxes), AXES))
    abar = np.zeros(len(boxes))
    for z, (t0, t1, h0, h1, w0, w1) in enumerate(boxes):
        X = A[t0:t1, h0:h1, w0:w1, :]
        for a in range(AXES):
            u[z, a] = line_variance_sum(X, a)
        abar[z] = X.mean()
    return u, abar


def _share(x: np.ndarray) -> np.ndarray:
    """x / sum(x) per row, with 0/0 := 0."""
    s = x.sum(axis=1, keepdims=True)
    out = np.zeros_like(x)
    np.divide(x, s, out=out, where=s > 0)
    return out


def zone_axis_scores(v, u, abar) -> np.ndarray:
    """S[Z, 3] = v_a / sum v + w u_a / sum u, w = abar / max abar (R4)."""
    amax = abar.max() if abar.size else 0.0
    w = abar / amax if amax > 0 else np.zeros_like(abar)
    return _share(v) + w[:, None] * _share(u)


def shape_costs(S, shapes) -> np.ndarray:
    """cost[Z, n_shapes] = sum_a S_a log2(e_a) (R4)."""
    logs = np.log2(np.asarray(shapes, dtype=np.float64))  # [n_shapes, 3]
    return S @ logs.T


def choose_shapes(S, shapes) -> np.ndarray:
    """Least-cost shape per zone, lowest index on ties, compared in fp32 (R4)."""
    c = shape_costs(S, shapes).astype(np.float32)
    return np.argmin(c, axis=1).astype(np.int32)  # argmin returns the first minimum


def block_permutation(grid, zext, zone_shape, shapes) -> np.ndarray:
    """perm[r] = raster index of the token at block-order position r (R5)."""
    T, H, W = grid
    out = []
    for z, (t0, t1, h0, h1, w0, w1) in enumerate(zone_boxes(grid, zext)):
        et, eh, ew = shapes[int(zone_shape[z])]
        for a in range(t0, t1, et):
            for b in range(h0, h1, eh):
                for c in range(w0, w1, ew):
                    tt = np.arange(a, min(a + et, t1))[:, None, None]
                    hh = np.arange(b, min(b + eh, h1))[None, :, None]
                    ww = np.arange(c, min(c + ew, w1))[None, None, :]
                    out.append(((tt * H + hh) * W + ww).reshape(-1))
    return np.concatenate(out).astype(np.int64)


def zone_token_counts(grid, zext) -> np.ndarray:
    """Tokens of every zone, raster zone order (R1)."""
    return np.array([(t1 - t0) * (h1 - h0) * (w1 - w0) for t0, t1, h0, h1, w0, w1 in zone_boxes(grid, zext)],
                    dtype=np.int64)


def block_permutation_chunked(grid, zext, zone_shape, shapes, B):
    """Zone-chunked blocks, the alternative reading of R5: the same token order as
    block_permutation, but every zone's run is cut into B-token blocks of its own (the
    last one short), so that no block holds tokens of two zones.

    Returned in a padded block order: each zone's run is followed by -1 entries up to a
    multiple of B, so block b is positions [b B, (b + 1) B) and its blen[b] tokens are
    the first ones.  Returns (perm_padded [Np] with -1 for padding, blen [nb])."""
    perm = block_permutation(grid, zext, zone_shape, shapes)
    out, blen, off = [], [], 0
    for n in zone_token_counts(grid, zext):
        run = perm[off:off + n]
        off += n
        nblk = -(-int(n) // B)
        padded = np.full(nblk * B, -1, dtype=np.int64)
        padded[:n] = run
        out.append(padded)
        blen.extend(min(B, int(n) - k * B) for k in range(nblk))
    return np.concatenate(out), np.array(blen, dtype=np.int64)


def zone_shapes(feature_chunks, a2v, grid, zext, shapes):
    """Step 1 of the path: (zone_shape[Z], perm[N], details) from V and the A2V field."""
    v = zone_video_variation(feature_chunks, grid, zext)
    u, abar = zone_a2v_coupling(a2v, grid, zext)
    S = zone_axis_scores(v, u, abar)
    zs = choose_shapes(S, shapes)
    perm = block_permutation(grid, zext, zs, shapes)
    return zs, perm, {"v": v, "u": u, "abar": abar, "S": S, "cost": shape_costs(S, shapes)}


# ----------------------------------------------------------------------- pool + score
def block_lengths(N: int, B: int) -> np.ndarray:
    nb = -(-N // B)
    lens = np.full(nb, B, dtype=np.int64)
    lens[-1] = N - B * (nb - 1)
    return lens


def block_mean(X_blk: np.ndarray, B: int, blen=None) -> np.ndarray:
    """Xbar[h, b, :] = mean over the tokens of block b of X_blk[:, h, :] (R6).

    X_blk is [N, Hh, d] in block order; with blen (zone-chunked blocks) block b is the
    first blen[b] rows of positions [b B, (b + 1) B).
    """
    N, Hh, d = X_blk.shape
    nb = -(-N // B)
    out = np.empty((Hh, nb, d))
    for b in range(nb):
        e = (b + 1) * B if blen is None else b * B + int(blen[b])
        out[:, b, :] = np.asarray(X_blk[b * B:e], dtype=np.float64).mean(axis=0)
    return out


def block_scores(qbar: np.ndarray, kbar: np.ndarray) -> np.ndarray:
    """S[h, i, j] = qbar[h, i] . kbar[h, j] / sqrt(d) (R6)."""
    d = qbar.shape[-1]
    return np.einsum("hid,hjd->hij", qbar, kbar) / math.sqrt(d)


def pool_score(Q, K, perm, B):
    """Step 2: block-order gather, block means and block scores.

    Q, K are [N, Hh, d] in raster order; returns (Qbar, Kbar, scores).
    """
    Qb = np.asarray(Q)[perm]
    Kb = np.asarray(K)[perm]
    qbar = block_mean(Qb, B)
    kbar = block_mean(Kb, B)
    return qbar, kbar, block_scores(qbar, kbar)


# --------------------------------------------------------------------------- select
def keep_count_topk(nb: int, sparsity: float) -> int:
    """k = ceil((1 - s) nb), at least 1 and at most nb; the 1e-9 absorbs fp error when
    (1 - s) nb is an integer (R7)."""
    return int(min(nb, max(1, math.ceil((1.0 - sparsity) * nb - 1e-9))))


def descending_order(s: np.ndarray) -> np.ndarray:
    """Block indices by score, largest first; equal scores by smaller index (R7)."""
    return np.lexsort((np.arange(s.size), -s))


def select_row(s_row, sparsity: float, cdf_tau: float):
    """Kept blocks of one query block, ascending, and the pair (k, m) (R7).

    The decision is taken on the row as stored (fp32 scores); the softmax mass is
    accumulated in fp64.
    """
    s = np.asarray(s_row, dtype=np.float32).astype(np.float64)
    nb = s.size
    order = descending_order(s)
    k = keep_count_topk(nb, sparsity)
    p = np.exp(s - s.max())
    p /= p.sum()
    cum = np.cumsum(p[order])
    hit = np.nonzero(cum >= cdf_tau)[0]
    m = int(hit[0]) + 1 if hit.size else nb
    r = max(k, m)
    return np.sort(order[:r]), k, m


def select(scores, sparsity: float, cdf_tau: float):
    """Step 3: (counts[Hh, nb], idx[Hh, nb, nb]) with ascending kept indices; unused
    entries are -1."""
    Hh, nb, _ = scores.shape
    counts = np.zeros((Hh, nb), dtype=np.int32)
    idx = np.full((Hh, nb, nb), -1, dtype=np.int32)
    for h in range(Hh):
        for i in range(nb):
            kept, _, _ = select_row(scores[h, i], sparsity, cdf_tau)
            counts[h, i] = kept.size
            idx[h, i, : kept.size] = kept
    return counts, idx


# ------------------------------------------------------------------------ attention
def block_rows(j, B: int, N: int, blen=None) -> np.ndarray:
    """Token positions (block order) of block j: the B-token chunk (the last one short),
    or the first blen[j] positions of the chunk for zone-chunked blocks."""
    e = min((j + 1) * B, N) if blen is None else j * B + int(blen[j])
    return np.arange(j * B, e)


def kept_tokens(kept_blocks, B: int, N: int, blen=None) -> np.ndarray:
    """Token positions (block order) covered by a list of blocks."""
    if len(kept_blocks) == 0:
        return np.zeros(0, dtype=np.int64)
    return np.concatenate([block_rows(int(j), B, N, blen) for j in kept_blocks])


def attention_row_block(q, Kc, Vc, scale):
    """Softmax attention of the rows q [M, d] over keys Kc, values Vc: (O, LSE) (R8)."""
    if Kc.shape[0] == 0:
        return np.zeros((q.shape[0], Vc.shape[1])), np.full(q.shape[0], -np.inf)
    S = (q @ Kc.T) * scale
    m = S.max(axis=1, keepdims=True)
    P = np.exp(S - m)
    l = P.sum(axis=1, keepdims=True)
    return (P @ Vc) / l, (m + np.log(l))[:, 0]


def bsa_forward(Qb, Kb, Vb, counts, idx, B, heads=None, qblocks=None, blen=None):
    """Step 4: O[N, Hh, d] and LSE[Hh, N] over the kept blocks (R8).

    Inputs are in block order.  ``heads`` / ``qblocks`` restrict the work to a
    sample; rows outside it are left as NaN.  With ``blen`` (zone-chunked blocks in a
    padded block order) only the first blen[b] positions of block b are tokens; padding
    positions are neither queries nor keys and stay NaN.
    """
    N, Hh, d = Qb.shape
    nb = -(-N // B)
    scale = 1.0 / math.sqrt(d)
    O = np.full((N, Hh, d), np.nan)
    LSE = np.full((Hh, N), np.nan)
    for h in (range(Hh) if heads is None else heads):
        for i in (range(nb) if qblocks is None else qblocks):
            rows = block_rows(i, B, N, blen)
            cols = kept_tokens(idx[h, i, : counts[h, i]], B, N, blen)
            o, lse = attention_row_block(np.asarray(Qb[rows, h], np.float64),
                                         np.asarray(Kb[cols, h], np.float64),
                                         np.asarray(Vb[cols, h], np.float64), scale)
            O[rows, h] = o
            LSE[h, rows] = lse
    return O, LSE


def a2v_field(Qv, Ka, Va, rows=None):
    """The A2V field (R9), from paragraph 1 of the page's block-construction section.

    Qv [N, Hh, d] video queries, Ka / Va [M, Hh, d] audio keys and values.  For every
    video token n (or only ``rows``): O[n, h] = softmax_m(Qv[n,h] . Ka[m,h] / sqrt(d))
    weighted sum of Va[m, h]; a2v[n] = sqrt(sum_h |O[n, h]|^2).  Returns (a2v, O) for
    the rows taken, O as [rows, Hh, d].
    """
    N, Hh, d = Qv.shape
    take = np.arange(N) if rows is None else np.asarray(rows)
    scale = 1.0 / math.sqrt(d)
    O = np.zeros((len(take), Hh, d))
    for h in range(Hh):
        o, _ = attention_row_block(np.asarray(Qv[take, h], np.float64), np.asarray(Ka[:, h], np.float64),
                                   np.asarray(Va[:, h], np.float64), scale)
        O[:, h] = o
    return np.sqrt((O * O).sum(axis=(1, 2))), O


def bsa_backward(Qb, Kb, Vb, O, dO, LSE, counts, idx, B, heads=None, qblocks=None, blen=None):
    """Step 5: dQ, dK, dV for the same kept lists (R8).

    P = exp(S - LSE), dV = P^T dO, dP = dO V^T, D = rowsum(dO * O),
    dS = P * (dP - D), dQ = dS K / sqrt(d), dK = dS^T Q / sqrt(d).
    ``heads`` / ``qblocks`` restrict the work to the contributions of a sample of
    query blocks (dK and dV then hold only those contributions).  ``blen`` as in
    bsa_forward (padding positions get zero gradients).
    """
    N, Hh, d = Qb.shape
    nb = -(-N // B)
    scale = 1.0 / math.sqrt(d)
    dQ = np.zeros((N, Hh, d))
    dK = np.zeros((N, Hh, d))
    dV = np.zeros((N, Hh, d))
    for h in (range(Hh) if heads is None else heads):
        for i in (range(nb) if qblocks is None else qblocks):
            rows = block_rows(i, B, N, blen)
            cols = kept_tokens(idx[h, i, : counts[h, i]], B, N, blen)
            if cols.size == 0:
                continue
            q = np.asarray(Qb[rows, h], np.float64)
            kc = np.asarray(Kb[cols, h], np.float64)
            vc = np.asarray(Vb[cols, h], np.float64)
            do = np.asarray(dO[rows, h], np.float64)
            o = np.asarray(O[rows, h], np.float64)
            P = np.exp(q @ kc.T * scale - np.asarray(LSE[h, rows], np.float64)[:, None])
            dV[cols, h] += P.T @ do
            dP = do @ vc.T
            D = (do * o).sum(axis=1)
            dS = P * (dP - D[:, None])
            dQ[rows, h] = dS @ kc * scale
            dK[cols, h] += dS.T @ q * scale
    return dQ, dK, dV


def transpose_lists(counts, idx):
    """For each (h, key block j): the query blocks i whose kept list holds j, ascending."""
    Hh, nb = counts.shape
    out = [[[] for _ in range(nb)] for _ in range(Hh)]
    for h in range(Hh):
        for i in range(nb):
            for j in idx[h, i, : counts[h, i]]:
                out[h][int(j)].append(i)
    return out


def bsa_backward_sampled(Qb, Kb, Vb, dO, counts, idx, B, h, qblocks, kblocks, tlists=None):
    """dQ of the query blocks ``qblocks`` and dK, dV of the key blocks ``kblocks`` of head h.

    Every query block that touches a sampled key block is re-run forward here
    (O, LSE of the oracle itself), so nothing from another implementation enters.
    Returns dicts block -> array [len, d].
    """
    N, Hh, d = Qb.shape
    scale = 1.0 / math.sqrt(d)
    tl = tlists if tlists is not None else transpose_lists(counts[h:h + 1], idx[h:h + 1])[0]
    need = set(qblocks)
    for j in kblocks:
        need.update(tl[j])
    dq, dk, dv = {}, {}, {}
    for j in kblocks:
        n = min((j + 1) * B, N) - j * B
        dk[j] = np.zeros((n, d))
        dv[j] = np.zeros((n, d))
    for i in sorted(need):
        rows = np.arange(i * B, min((i + 1) * B, N))
        kept = idx[h, i, : counts[h, i]]
        cols = kept_tokens(kept, B, N)
        if cols.size == 0:
            if i in qblocks:
                dq[i] = np.zeros((rows.size, d))
            continue
        q = np.asarray(Qb[rows, h], np.float64)
        kc = np.asarray(Kb[cols, h], np.float64)
        vc = np.asarray(Vb[cols, h], np.float64)
        do = np.asarray(dO[rows, h], np.float64)
        o, lse = attention_row_block(q, kc, vc, scale)
        P = np.exp(q @ kc.T * scale - lse[:, None])
        dP = do @ vc.T
        D = (do * o).sum(axis=1)
        dS = P * (dP - D[:, None])
        if i in qblocks:
            dq[i] = dS @ kc * scale
        off = 0
        for j in kept:
            n = min((int(j) + 1) * B, N) - int(j) * B
            if int(j) in dk:
                dv[int(j)] += P[:, off:off + n].T @ do
                dk[int(j)] += dS[:, off:off + n].T @ q * scale
            off += n
    return dq, dk, dv


# -------------------------------------------------- attention broadcast (PAB)
def attn_mse(A, B):
    """mse[h] = mean over tokens n and channels c of (A[n, h, c] - B[n, h, c])^2.

    The difference measure between the attention outputs of two diffusion steps that
    the "Real-time video generation with pyramid attention broadcast" page uses to
    choose broadcast ranges (method section: MSE between consecutive steps' attention
    outputs).  A, B are [N, Hh, d].
    """
    D = np.asarray(A, np.float64) - np.asarray(B, np.float64)
    return (D * D).mean(axis=(0, 2))


def pab_schedule(n_steps: int, broadcast_range: int, window=(0.15, 0.85)):
    """Per diffusion step: True where attention is computed, False where the previous
    computed output is broadcast (reused).

    Same page: the difference between consecutive steps' attention outputs is
    U-shaped, small through the middle 70% of the steps, so outputs computed there are
    broadcast to the following steps.  Readings: the middle window is steps
    [round(0.15 T), round(0.85 T)); inside it attention is computed at the window's
    first step and then every (range + 1) steps, each computed output serving the
    `range` steps after it; every step outside the window computes.
    """
    lo, hi = int(round(window[0] * n_steps)), int(round(window[1] * n_steps))
    out = []
    for t in range(n_steps):
        out.append(not (lo <= t < hi) or (t - lo) % (broadcast_range + 1) == 0)
    return out
