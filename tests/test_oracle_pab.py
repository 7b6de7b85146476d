"""Pins of the oracle's attention-broadcast pieces against closed forms: the MSE of
two outputs and the broadcast schedule (Pyramid Attention Broadcast page, method)."""
import numpy as np

from oracle import prism_oracle as po


def test_attn_mse_closed_forms():
    rng = np.random.default_rng(0)
    A = rng.normal(size=(37, 3, 8))
    assert np.all(po.attn_mse(A, A) == 0)
    c = np.array([0.5, -2.0, 3.0])
    np.testing.assert_allclose(po.attn_mse(A + c[None, :, None], A), c ** 2, rtol=1e-12)
    # per head, independent of the other heads; symmetric; scales quadratically
    B = rng.normal(size=A.shape)
    m = po.attn_mse(A, B)
    B2 = B.copy()
    B2[:, 1] = A[:, 1]
    assert m[1] > 0 and po.attn_mse(A, B2)[1] == 0 and po.attn_mse(A, B2)[0] == m[0]
    np.testing.assert_allclose(po.attn_mse(B, A), m)
    np.testing.assert_allclose(po.attn_mse(3 * A, 3 * B), 9 * m)
    # brute force on one head
    brute = sum((A[n, 2, k] - B[n, 2, k]) ** 2 for n in range(37) for k in range(8)) / (37 * 8)
    np.testing.assert_allclose(m[2], brute, rtol=1e-12)


def test_pab_schedule_closed_forms():
    # 30 steps, range 2: window [4, 26) (round(4.5) = 4, round(25.5) = 26 by banker's rounding)
    s = po.pab_schedule(30, 2)
    computed = [t for t, c in enumerate(s) if c]
    assert computed == [0, 1, 2, 3] + list(range(4, 26, 3)) + [26, 27, 28, 29]
    # range 0 computes every step; the window's first step always computes
    assert all(po.pab_schedule(30, 0))
    s = po.pab_schedule(50, 4)
    lo, hi = 8, 42
    assert s[lo] and not any(s[lo + 1:lo + 5]) and s[lo + 5]
    assert all(s[:lo]) and all(s[hi:])
    # every broadcast step follows a computed step at most `range` steps earlier
    for n, r in ((30, 2), (50, 4), (7, 1), (100, 9)):
        s = po.pab_schedule(n, r)
        last = None
        for t, c in enumerate(s):
            if c:
                last = t
            else:
                assert last is not None and t - last <= r


def test_product_schedule_equals_oracle():
    # the library-side schedule (host logic) against the oracle's restatement
    from audio_diffusion_dits_zone_b300 import pab

    for n, r in ((30, 2), (50, 4), (7, 1), (100, 9), (30, 0), (1, 3)):
        assert pab.schedule(n, r) == po.pab_schedule(n, r)
