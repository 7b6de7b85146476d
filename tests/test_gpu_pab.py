"""Attention broadcast across diffusion steps on the GPU: the library's per-head MSE of
two attention outputs against the oracle's, on ragged sizes, strided head views and
both dtypes; identical inputs give exactly 0."""
import numpy as np
import pytest
import torch

from audio_diffusion_dits_zone_b300 import prism as P
from audio_diffusion_dits_zone_b300 import synth
from oracle import prism_oracle as po

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("N,Hh,d,dtype", [(1000, 3, 128, "bf16"), (75600, 40, 128, "bf16"), (333, 2, 64, "f32"),
                                          (7, 5, 128, "bf16"), (129, 2, 24, "bf16")])
def test_attn_mse_matches_oracle(N, Hh, d, dtype):
    rng = np.random.default_rng(N + d)
    A = rng.normal(size=(N, Hh, d)).astype(np.float32)
    B = (A + rng.normal(scale=0.1, size=A.shape) * rng.uniform(0, 2, size=(1, Hh, 1))).astype(np.float32)
    if dtype == "bf16":
        A, B = synth.to_bf16(A), synth.to_bf16(B)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    a, b = (torch.from_numpy(x).cuda().to(tdt) for x in (A, B))
    mse = torch.empty(Hh, device="cuda")
    P.prism_attn_mse(a, b, mse)
    assert P.status_check() == 0
    ref = po.attn_mse(A, B)
    np.testing.assert_allclose(mse.cpu().numpy(), ref, rtol=1e-5)
    P.prism_attn_mse(a, a, mse)
    assert np.all(mse.cpu().numpy() == 0)


def test_attn_mse_on_head_views():
    # a group of heads of a larger tensor: pointer offset, token row stride of the whole
    rng = np.random.default_rng(5)
    A = synth.to_bf16(rng.normal(size=(500, 8, 128)).astype(np.float32))
    B = synth.to_bf16(rng.normal(size=(500, 8, 128)).astype(np.float32))
    a, b = (torch.from_numpy(x).cuda().bfloat16() for x in (A, B))
    mse = torch.empty(3, device="cuda")
    P.prism_attn_mse(a[:, 2:5], b[:, 2:5], mse)
    assert P.status_check() == 0
    np.testing.assert_allclose(mse.cpu().numpy(), po.attn_mse(A[:, 2:5], B[:, 2:5]), rtol=1e-5)


def _trajectory_case():
    from audio_diffusion_dits_zone_b300.pipeline import PrismLayer

    wl = synth.Workload("pab", 90, (3, 18, 32), 2, 128, "bf16", (3, 9, 16), 128, synth.SHAPES_128, 0.75, 0.2, 1,
                        3.0, (44, 42, 42), "fwd")
    hs = range(wl.heads)
    clean = {t: np.stack(synth.gen_heads(wl, t, hs), axis=1) for t in (synth.Q_ID, synth.K_ID, synth.V_ID)}
    noise = {t: np.stack([synth.gen_noise_head(wl, t, h) for h in hs], axis=1) for t in clean}
    a2v = synth.gen_a2v(wl)

    def step_inputs(t, n):
        return [synth.round_inputs(wl, synth.trajectory_blend(clean[x], noise[x], t, n)) for x in
                (synth.Q_ID, synth.K_ID, synth.V_ID)]

    layer = PrismLayer(wl, "cuda", train=False)
    layer.a2v.copy_(torch.from_numpy(a2v))
    return wl, layer, step_inputs, a2v


def _oracle_step(wl, Q, K, V, a2v):
    zs, perm, _ = po.zone_shapes([V.reshape(wl.N, -1)], a2v, wl.grid, wl.zone, wl.shapes)
    _, _, S = po.pool_score(Q.astype(np.float64), K.astype(np.float64), perm, wl.block)
    counts, idx = po.select(S, wl.sparsity, wl.cdf_tau)
    return perm, counts, idx


@pytest.mark.parametrize("mode", ["outputs", "lists"])
def test_broadcast_layer_follows_the_schedule(mode):
    from audio_diffusion_dits_zone_b300 import pab
    from parity import attn_close

    n = 7
    wl, layer, step_inputs, a2v = _trajectory_case()
    bl = pab.BroadcastLayer(layer, n, 1, mode)
    assert bl.plan == [True, True, False, True, False, True, True]
    last = None  # the oracle's selection of the last computed step, and its output
    for t in range(n):
        Q, K, V = step_inputs(t, n)
        for dst, x in ((layer.q, Q), (layer.k, K), (layer.v, V)):
            dst.copy_(torch.from_numpy(x).to(torch.bfloat16))
        before = layer.o_blk.clone()
        computed = bl.run_step(t)
        assert P.status_check() == 0
        assert computed == bl.plan[t]
        got = layer.o_blk.float().cpu().numpy()
        if computed:
            perm, counts, idx = _oracle_step(wl, Q, K, V, a2v)
            assert np.array_equal(layer.perm.cpu().numpy(), perm)
            O, _ = po.bsa_forward(*(x[perm].astype(np.float64) for x in (Q, K, V)), counts, idx, wl.block)
            attn_close(got, O, what=f"step {t}")
            last = (perm, counts, idx)
        elif mode == "outputs":
            assert torch.equal(layer.o_blk, before)          # broadcast: nothing recomputed
        else:
            perm, counts, idx = last                          # the held selection, this step's Q, K, V
            O, _ = po.bsa_forward(*(x[perm].astype(np.float64) for x in (Q, K, V)), counts, idx, wl.block)
            attn_close(got, O, what=f"step {t} (lists held)")


def test_calibration_curve_matches_oracle():
    from audio_diffusion_dits_zone_b300 import pab

    n = 5
    wl, layer, step_inputs, a2v = _trajectory_case()

    def set_inputs(t):
        for dst, x in zip((layer.q, layer.k, layer.v), step_inputs(t, n)):
            dst.copy_(torch.from_numpy(x).to(torch.bfloat16))

    curve = pab.calibrate(layer, set_inputs, n).cpu().numpy()
    assert P.status_check() == 0
    Q, K, V = step_inputs(0, n)
    perm, counts, idx = _oracle_step(wl, Q, K, V, a2v)
    outs = []
    for t in range(n):
        Q, K, V = step_inputs(t, n)
        O, _ = po.bsa_forward(*(x[perm].astype(np.float64) for x in (Q, K, V)), counts, idx, wl.block)
        outs.append(synth.to_bf16(O.astype(np.float32)))
    ref = np.stack([po.attn_mse(outs[t], outs[t - 1]) for t in range(1, n)])
    # the outputs are bf16 on both sides; their MSEs agree to the bf16 rounding of O
    np.testing.assert_allclose(curve, ref, rtol=0.05, atol=1e-5)
