"""Pins for the oracle's zone statistics, shape choice and block permutation.

Closed forms (linear ramps have a known line variance), special cases that fix
the shape choice, a brute-force line enumeration on a tiny grid, and
hand-worked permutations (tests/golden/perm_cases.json).
"""
import json
import os

import numpy as np
import pytest

from oracle import prism_oracle as po

SH128 = ((1, 8, 16), (2, 8, 8), (4, 4, 8), (8, 4, 4))
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def ramp_feature(grid, axis, alphas):
    """F[t,h,w,c] = alpha_c * coord_axis + c: linear along one axis only."""
    T, H, W = grid
    coords = np.meshgrid(np.arange(T), np.arange(H), np.arange(W), indexing="ij")[axis]
    F = coords[..., None] * np.asarray(alphas)[None, None, None, :] + np.arange(len(alphas))
    return F.reshape(T * H * W, len(alphas)).astype(np.float64)


@pytest.mark.parametrize("axis", [0, 1, 2])
def test_ramp_variance_closed_form(axis):
    # Population variance of alpha*{0..L-1} is alpha^2 (L^2 - 1) / 12; zones clip at the edge.
    grid, zext = (5, 8, 16), (3, 3, 8)
    alphas = [0.5, -1.25, 2.0]
    v = po.zone_video_variation([ramp_feature(grid, axis, alphas)], grid, zext)
    mean_a2 = np.mean(np.square(alphas))
    for z, box in enumerate(po.zone_boxes(grid, zext)):
        L = box[2 * axis + 1] - box[2 * axis]
        expect = np.zeros(3)
        expect[axis] = mean_a2 * (L * L - 1) / 12.0
        np.testing.assert_allclose(v[z], expect, rtol=1e-12, atol=1e-12)


def test_zone_boxes_clip_and_order():
    boxes = po.zone_boxes((21, 68, 120), (3, 9, 16))
    assert len(boxes) == 7 * 8 * 8
    assert boxes[0] == (0, 3, 0, 9, 0, 16)
    assert boxes[7] == (0, 3, 0, 9, 112, 120)      # last w zone clipped to 8
    assert boxes[8] == (0, 3, 9, 18, 0, 16)        # raster order: w fastest, then h
    assert boxes[-1] == (18, 21, 63, 68, 112, 120)  # h clipped to 5
    assert len(po.zone_boxes((21, 45, 80), (3, 9, 16))) == 175
    assert len(po.zone_boxes((21, 90, 160), (3, 9, 16))) == 700


def test_brute_force_line_variance():
    # Enumerate every line of every zone with plain loops on a tiny random grid.
    rng = np.random.default_rng(3)
    grid, zext = (4, 3, 5), (3, 2, 4)
    T, H, W = grid
    F = rng.normal(size=(T * H * W, 2))
    v = po.zone_video_variation([F[:, :1], F[:, 1:]], grid, zext)
    F4 = F.reshape(T, H, W, 2)
    for z, (t0, t1, h0, h1, w0, w1) in enumerate(po.zone_boxes(grid, zext)):
        ranges = [range(t0, t1), range(h0, h1), range(w0, w1)]
        for a in range(3):
            others = [ranges[b] for b in range(3) if b != a]
            tot, nlines = 0.0, 0
            for c in range(2):
                for x in others[0]:
                    for y in others[1]:
                        vals = []
                        for p in ranges[a]:
                            idx = [0, 0, 0]
                            idx[a] = p
                            idx[[b for b in range(3) if b != a][0]] = x
                            idx[[b for b in range(3) if b != a][1]] = y
                            vals.append(F4[idx[0], idx[1], idx[2], c])
                        mu = sum(vals) / len(vals)
                        tot += sum((q - mu) ** 2 for q in vals) / len(vals)
                        if c == 0:
                            nlines += 1
            assert v[z, a] == pytest.approx(tot / nlines / 2, rel=1e-12, abs=1e-15)


@pytest.mark.parametrize("axis,expect", [(0, 0), (2, 3), (1, 2)])
def test_shape_choice_single_axis(axis, expect):
    # Only axis `axis` varies: S = e_axis; cost of (et,eh,ew) is log2 e_axis.
    # t -> (1,8,16); w -> (8,4,4); h -> costs 3,3,2,2 -> tie -> lowest index (4,4,8).
    grid, zext = (6, 16, 32), (3, 8, 16)
    F = ramp_feature(grid, axis, [1.0, 0.3])
    a2v = np.ones(np.prod(grid))
    zs, perm, det = po.zone_shapes([F], a2v, grid, zext, SH128)
    assert np.all(det["u"] == 0)
    assert np.all(zs == expect)


def test_constant_fields_tie_to_shape_zero():
    grid, zext = (6, 16, 32), (3, 8, 16)
    N = int(np.prod(grid))
    zs, _, det = po.zone_shapes([np.full((N, 4), 0.75)], np.full(N, 0.5), grid, zext, SH128)
    assert np.all(det["S"] == 0)
    assert np.all(zs == 0)


def test_a2v_constant_along_t_has_no_t_coupling():
    T, H, W = 6, 16, 32
    hh, ww = np.meshgrid(np.arange(H), np.arange(W), indexing="ij")
    bump = np.exp(-((hh - 5.0) ** 2 + (ww - 20.0) ** 2) / 18.0)
    a2v = np.broadcast_to(bump, (T, H, W)).reshape(-1)
    u, abar = po.zone_a2v_coupling(a2v, (T, H, W), (3, 8, 16))
    # exactly 0 up to the rounding of a mean of equal values
    assert np.all(u[:, 0] <= 1e-12 * u[:, 1:].sum(axis=1))
    assert np.all(u[:, 1:].sum(axis=1) > 0)
    assert np.all(abar > 0)


def test_a2v_drives_shape_when_video_is_flat():
    # Flat video, A2V varying along w only, in proportion to the zone: S = w * (0, 0, 1).
    T, H, W = 6, 16, 32
    ww = np.broadcast_to(np.arange(W, dtype=np.float64), (T, H, W)).reshape(-1)
    a2v = 1.0 + 0.01 * ww
    zs, _, det = po.zone_shapes([np.zeros((T * H * W, 2))], a2v, (T, H, W), (3, 8, 16), SH128)
    np.testing.assert_allclose(det["S"][:, :2], 0.0, atol=1e-20)   # up to mean-of-equal rounding
    np.testing.assert_allclose(det["S"][:, 2], det["abar"] / det["abar"].max())
    assert np.all(zs == 3)


def test_weight_scales_a2v_term():
    # Video varies along t in every zone; A2V varies along w in one zone only, with a
    # large mean there.  That zone's S mixes both terms with weight 1; others keep (1,0,0).
    T, H, W = 3, 8, 32
    grid, zext = (T, H, W), (3, 8, 16)
    F = ramp_feature(grid, 0, [1.0])
    a2v = np.zeros((T, H, W))
    a2v[:, :, 16:] = 5.0 + np.arange(16)[None, None, :]
    zs, _, det = po.zone_shapes([F], a2v.reshape(-1), grid, zext, SH128)
    np.testing.assert_allclose(det["S"][0], [1.0, 0.0, 0.0])
    np.testing.assert_allclose(det["S"][1], [1.0, 0.0, 1.0])
    # zone 1 costs: (1,8,16) 4, (2,8,8) 4, (4,4,8) 5, (8,4,4) 5 -> tie -> shape 0
    assert list(zs) == [0, 0]


def test_permutation_golden():
    with open(os.path.join(GOLDEN, "perm_cases.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        perm = po.block_permutation(tuple(c["grid"]), tuple(c["zone"]), c["zone_shape"],
                                    [tuple(s) for s in c["shapes"]])
        assert perm.tolist() == c["perm"]


@pytest.mark.parametrize("grid,zext", [((21, 45, 80), (3, 9, 16)), ((21, 68, 120), (3, 9, 16)),
                                       ((5, 8, 16), (5, 4, 8))])
def test_permutation_bijection_and_tiles(grid, zext):
    T, H, W = grid
    Z = len(po.zone_boxes(grid, zext))
    rng = np.random.default_rng(1)
    zs = rng.integers(0, 4, size=Z)
    shapes = SH128 if grid[0] > 5 else ((1, 8, 8), (2, 4, 8), (4, 4, 4), (8, 2, 4))
    perm = po.block_permutation(grid, zext, zs, shapes)
    assert perm.size == T * H * W
    assert np.array_equal(np.sort(perm), np.arange(T * H * W))
    # every zone's tokens are one contiguous run of the block order
    pos = np.empty_like(perm)
    pos[perm] = np.arange(perm.size)
    start = 0
    for (t0, t1, h0, h1, w0, w1) in po.zone_boxes(grid, zext):
        t, h, w = np.meshgrid(np.arange(t0, t1), np.arange(h0, h1), np.arange(w0, w1), indexing="ij")
        p = np.sort(pos[((t * H + h) * W + w).reshape(-1)])
        assert p[0] == start and p[-1] == start + p.size - 1
        start += p.size
