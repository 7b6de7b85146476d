"""Pins of the oracle's A2V field (cross-attention feature norm) to what the
mathematics fixes, independently of the oracle's own code path.

"Prism: dynamic sparse attention for 2K joint video-audio generation training",
section "Region-adapted block construction", paragraph 1 (the feature norm of the
audio-to-video cross-attention), read as: per head softmax attention of each video
token over all audio tokens, then the L2 norm of the token's output over all heads.
"""
import math

import numpy as np

import oracle as po


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def test_single_audio_token_gives_its_value_everywhere():
    # one key: every softmax weight is 1, so O[n, h] = Va[0, h] for every token
    Qv, Ka, Va = _rand((50, 3, 8), 1), _rand((1, 3, 8), 2), _rand((1, 3, 8), 3)
    a2v, O = po.a2v_field(Qv, Ka, Va)
    assert np.allclose(O, np.broadcast_to(Va[0], O.shape), rtol=0, atol=1e-14)
    assert np.allclose(a2v, np.linalg.norm(Va[0]), rtol=1e-14)


def test_equal_keys_or_zero_queries_average_the_values():
    Va = _rand((7, 2, 8), 4)
    mean = Va.mean(axis=0)  # [Hh, d]
    Ka_same = np.broadcast_to(_rand((1, 2, 8), 5), (7, 2, 8)).copy()
    a2v, _ = po.a2v_field(_rand((20, 2, 8), 6), Ka_same, Va)
    assert np.allclose(a2v, np.linalg.norm(mean), rtol=1e-13)
    a2v0, _ = po.a2v_field(np.zeros((5, 2, 8)), _rand((7, 2, 8), 7), Va)
    assert np.allclose(a2v0, np.linalg.norm(mean), rtol=1e-13)


def test_two_audio_tokens_closed_form():
    # two keys: weight of key 0 = 1 / (1 + exp(s1 - s0)), s_m = q . k_m / sqrt(d)
    d = 16
    Qv, Ka, Va = _rand((9, 1, d), 8), _rand((2, 1, d), 9), _rand((2, 1, d), 10)
    a2v, O = po.a2v_field(Qv, Ka, Va)
    for n in range(9):
        s0 = float(Qv[n, 0] @ Ka[0, 0]) / math.sqrt(d)
        s1 = float(Qv[n, 0] @ Ka[1, 0]) / math.sqrt(d)
        w0 = 1.0 / (1.0 + math.exp(s1 - s0))
        o = w0 * Va[0, 0] + (1.0 - w0) * Va[1, 0]
        assert np.allclose(O[n, 0], o, rtol=1e-12, atol=1e-14)
        assert abs(a2v[n] - np.linalg.norm(o)) <= 1e-12 * max(1.0, np.linalg.norm(o))


def test_invariances():
    Qv, Ka, Va = _rand((30, 2, 8), 11), _rand((13, 2, 8), 12), _rand((13, 2, 8), 13)
    a2v, _ = po.a2v_field(Qv, Ka, Va)
    # permuting the audio tokens (keys and values together) changes nothing
    p = np.random.default_rng(14).permutation(13)
    assert np.allclose(po.a2v_field(Qv, Ka[p], Va[p])[0], a2v, rtol=1e-13)
    # a vector added to every key shifts each row's scores by a constant: softmax unchanged
    assert np.allclose(po.a2v_field(Qv, Ka + _rand((1, 2, 8), 15), Va)[0], a2v, rtol=1e-11)
    # values scaled by c scale the norm by |c|
    assert np.allclose(po.a2v_field(Qv, Ka, -2.5 * Va)[0], 2.5 * a2v, rtol=1e-13)
    # heads add in squares
    a0, _ = po.a2v_field(Qv[:, :1], Ka[:, :1], Va[:, :1])
    a1, _ = po.a2v_field(Qv[:, 1:], Ka[:, 1:], Va[:, 1:])
    assert np.allclose(a2v ** 2, a0 ** 2 + a1 ** 2, rtol=1e-12)


def test_brute_force_loops_on_a_tiny_case():
    Qv, Ka, Va = _rand((4, 2, 3), 16), _rand((5, 2, 3), 17), _rand((5, 2, 3), 18)
    a2v, _ = po.a2v_field(Qv, Ka, Va, rows=[0, 2, 3])
    for r, n in enumerate([0, 2, 3]):
        total = 0.0
        for h in range(2):
            e = [math.exp(sum(Qv[n, h, c] * Ka[m, h, c] for c in range(3)) / math.sqrt(3)) for m in range(5)]
            z = sum(e)
            for c in range(3):
                oc = sum(e[m] * Va[m, h, c] for m in range(5)) / z
                total += oc * oc
        assert abs(a2v[r] - math.sqrt(total)) <= 1e-12
