"""The seeded input module: determinism, shapes and the recipe's stated statistics."""
import numpy as np

from audio_diffusion_dits_zone_b300 import synth


def test_workload_sizes():
    w = synth.WORKLOADS
    assert (w["tiny"].N, w["tiny"].nb) == (640, 10)
    assert (w["720p"].N, w["720p"].nb) == (75600, 591)
    assert (w["1080p"].N, w["1080p"].nb) == (171360, 1339)
    assert (w["2k"].N, w["2k"].nb) == (302400, 2363)
    assert w["720p"].N - 128 * (w["720p"].nb - 1) == 80
    assert w["1080p"].N - 128 * (w["1080p"].nb - 1) == 96
    assert w["2k"].N - 128 * (w["2k"].nb - 1) == 64


def test_generators_are_deterministic_and_distinct():
    wl = synth.WORKLOADS["tiny"]
    a = synth.gen_head(wl, synth.Q_ID, 0)
    b = synth.gen_head(wl, synth.Q_ID, 0)
    c = synth.gen_head(wl, synth.Q_ID, 1)
    assert a.shape == (640, 64) and a.dtype == np.float32
    assert np.array_equal(a, b) and not np.allclose(a, c)
    assert np.array_equal(synth.gen_a2v(wl), synth.gen_a2v(wl))


def test_rope_preserves_pair_norms():
    wl = synth.WORKLOADS["tiny"]
    cos, sin = synth.rope_tables(wl.grid, wl.d, wl.rope_split)
    x = np.random.default_rng(0).normal(size=(wl.N, wl.d)).astype(np.float32)
    y = synth._apply_rope(x, cos, sin)
    np.testing.assert_allclose(x[:, 0::2] ** 2 + x[:, 1::2] ** 2, y[:, 0::2] ** 2 + y[:, 1::2] ** 2, rtol=1e-5)
    assert np.allclose(cos[0], 1) and np.allclose(sin[0], 0)   # token (0,0,0) is not rotated


def test_a2v_bump_peaks_near_one_and_bf16_rounding():
    wl = synth.WORKLOADS["720p"]
    a = synth.gen_a2v(wl)
    assert a.shape == (wl.N,) and 0.5 < a.max() <= 1.0 + 1e-6 and a.min() >= 0
    # bf16 spacing at 1 is 2^-7; halfway cases go to the even mantissa
    x = np.array([1.0078125, 1.00390625, 1.01171875, 3.14159], np.float32)
    assert synth.to_bf16(x).tolist() == [1.0078125, 1.0, 1.015625, 3.140625]
