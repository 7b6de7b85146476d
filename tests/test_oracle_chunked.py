"""Pins of the oracle's zone-chunked block layout (the alternative reading of the block
order: every zone cut into B-token blocks of its own): closed forms of the block
counts, the token order, no block across two zones, padding excluded from the block
means and from attention (brute force on the compacted tokens)."""
import numpy as np

from oracle import prism_oracle as po


def _zone_of_token(grid, zext):
    T, H, W = grid
    z = np.empty(T * H * W, np.int64)
    for k, (t0, t1, h0, h1, w0, w1) in enumerate(po.zone_boxes(grid, zext)):
        tt, hh, ww = np.meshgrid(np.arange(t0, t1), np.arange(h0, h1), np.arange(w0, w1), indexing="ij")
        z[((tt * H + hh) * W + ww).ravel()] = k
    return z


def test_chunked_720p_closed_form():
    grid, zext, B = (21, 45, 80), (3, 9, 16), 128
    Z = len(po.zone_boxes(grid, zext))
    zs = np.random.default_rng(0).integers(0, 4, Z)
    pp, blen = po.block_permutation_chunked(grid, zext, zs, ((1, 8, 16), (2, 8, 8), (4, 4, 8), (8, 4, 4)), B)
    # 175 zones of 3 x 9 x 16 = 432 tokens: blocks of 128, 128, 128, 48
    assert Z == 175 and blen.size == 700 and pp.size == 700 * 128
    assert np.array_equal(blen, np.tile([128, 128, 128, 48], 175))
    assert (pp >= 0).sum() == 21 * 45 * 80


def test_chunked_1080p_block_count():
    # 68 = 7 * 9 + 5 and 120 = 7 * 16 + 8: zones of 432, 240, 216 and 120 tokens, i.e.
    # 4, 2, 2 and 1 blocks; per t-plane 49 * 4 + 7 * 2 + 7 * 2 + 1 = 225 blocks
    grid, zext, B = (21, 68, 120), (3, 9, 16), 128
    zs = np.zeros(len(po.zone_boxes(grid, zext)), np.int64)
    pp, blen = po.block_permutation_chunked(grid, zext, zs, ((1, 8, 16),), B)
    assert blen.size == 7 * 225 and blen.sum() == 21 * 68 * 120 and pp.size == blen.size * B


def test_chunked_order_blocks_and_padding():
    rng = np.random.default_rng(3)
    for grid, zext, B, shapes in (((5, 8, 16), (5, 4, 8), 64, ((1, 8, 8), (2, 4, 8), (4, 4, 4), (8, 2, 4))),
                                  ((7, 20, 40), (3, 9, 16), 128, ((1, 8, 16), (2, 8, 8), (4, 4, 8), (8, 4, 4))),
                                  ((4, 10, 13), (3, 4, 5), 16, ((1, 2, 8), (2, 2, 4), (4, 2, 2)))):
        Z = len(po.zone_boxes(grid, zext))
        zs = rng.integers(0, len(shapes), Z)
        pp, blen = po.block_permutation_chunked(grid, zext, zs, shapes, B)
        # the same token order as the consecutive-chunk layout
        assert np.array_equal(pp[pp >= 0], po.block_permutation(grid, zext, zs, shapes))
        zone = _zone_of_token(grid, zext)
        counts = po.zone_token_counts(grid, zext)
        k = 0
        for z in range(Z):
            for m in range(-(-int(counts[z]) // B)):
                rows = pp[k * B:(k + 1) * B]
                assert blen[k] == min(B, counts[z] - m * B)
                assert np.all(rows[:blen[k]] >= 0) and np.all(rows[blen[k]:] == -1)
                assert np.all(zone[rows[:blen[k]]] == z)  # one zone per block
                k += 1
        assert k == blen.size


def test_chunked_means_and_attention_skip_padding():
    rng = np.random.default_rng(5)
    B, d = 16, 8
    blen = np.array([16, 5, 16, 9, 1])
    nb = blen.size
    N = nb * B
    valid = np.concatenate([np.arange(b * B, b * B + blen[b]) for b in range(nb)])
    X = rng.normal(size=(N, 2, d))
    Xp = X.copy()
    pad = np.setdiff1d(np.arange(N), valid)
    Xp[pad] = 1e9  # padding rows never count
    np.testing.assert_allclose(po.block_mean(Xp, B, blen)[:, 1], X[B:B + 5].mean(0))
    Q, K, V = (rng.normal(size=(N, 1, d)) for _ in range(3))
    for A in (Q, K, V):
        A[pad] = 1e3
    counts = np.array([[3, 1, 5, 2, 4]])
    idx = np.zeros((1, nb, nb), np.int64)
    lists = [[0, 1, 4], [1], [0, 1, 2, 3, 4], [2, 4], [0, 1, 3, 4]]
    for i, l in enumerate(lists):
        idx[0, i, : len(l)] = l
    O, L = po.bsa_forward(Q, K, V, counts, idx, B, blen=blen)
    for i, l in enumerate(lists):
        rows = np.arange(i * B, i * B + blen[i])
        cols = np.concatenate([np.arange(j * B, j * B + blen[j]) for j in l])
        S = Q[rows, 0] @ K[cols, 0].T / np.sqrt(d)
        P = np.exp(S - S.max(1, keepdims=True))
        np.testing.assert_allclose(O[rows, 0], (P / P.sum(1, keepdims=True)) @ V[cols, 0], rtol=1e-10, atol=1e-12)
        assert np.all(np.isnan(O[i * B + blen[i]:(i + 1) * B]))
    # uniform chunks with the short last block: the same as the consecutive layout
    blen_u = np.array([min(B, 70 - j * B) for j in range(5)])
    Qu, Ku, Vu = (rng.normal(size=(70, 1, d)) for _ in range(3))
    c2, i2 = counts, idx
    a = po.bsa_forward(Qu, Ku, Vu, c2, i2, B)[0]
    b = po.bsa_forward(Qu, Ku, Vu, c2, i2, B, blen=blen_u)[0]
    np.testing.assert_array_equal(a, b)
