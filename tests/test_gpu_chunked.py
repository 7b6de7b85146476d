"""Zone-chunked blocks on the GPU (every zone cut into B-token blocks of its own, padded
block order with per-block lengths) against the oracle: the padded permutation and the
block lengths exactly, block means and copies with padding, attention forward and
backward over blocks with padding (tensor-core and CUDA-core paths), and the whole
layer on the tiny workload."""
import numpy as np
import pytest
import torch

from audio_diffusion_dits_zone_b300 import prism as P
from audio_diffusion_dits_zone_b300 import synth
from audio_diffusion_dits_zone_b300.pipeline import PrismLayer
from oracle import prism_oracle as po
from parity import attn_close, check_lists

pytestmark = pytest.mark.gpu
dev = "cuda"


@pytest.mark.parametrize("grid,zext,B,shapes", [((5, 8, 16), (5, 4, 8), 64, synth.SHAPES_64),
                                                ((21, 68, 120), (3, 9, 16), 128, synth.SHAPES_128),
                                                ((4, 10, 13), (3, 4, 5), 16, ((1, 2, 8), (2, 2, 4), (4, 2, 2)))])
def test_perm_chunked_matches_oracle(grid, zext, B, shapes):
    Z = len(po.zone_boxes(grid, zext))
    zs = np.random.default_rng(Z).integers(0, len(shapes), Z).astype(np.int32)
    nb, np_ = P.prism_zone_chunked_size(grid, zext, B)
    pp = torch.full((np_,), 7, dtype=torch.int32, device=dev)
    bl = torch.empty(nb, dtype=torch.int32, device=dev)
    P.prism_zone_perm_chunked(torch.from_numpy(zs).to(dev), grid, zext, shapes, B, pp, bl)
    assert P.status_check() == 0
    opp, obl = po.block_permutation_chunked(grid, zext, zs, shapes, B)
    assert np.array_equal(pp.cpu().numpy(), opp) and np.array_equal(bl.cpu().numpy(), obl)


def chunked_case(N_grid=(6, 18, 32), zext=(3, 9, 16), heads=2, d=128, dtype="bf16", B=128, cid=91):
    shapes = synth.SHAPES_128 if B == 128 else synth.SHAPES_64
    split = (44, 42, 42) if d == 128 else (16, 24, 24)
    wl = synth.Workload("chunk", cid, N_grid, heads, d, dtype, zext, B, shapes, 0.75, 0.2, 1, 3.0, split, "fwd+bwd")
    Z = len(po.zone_boxes(N_grid, zext))
    zs = np.random.default_rng(cid).integers(0, len(shapes), Z)
    pp, blen = po.block_permutation_chunked(N_grid, zext, zs, shapes, B)
    return wl, pp, blen


@pytest.mark.parametrize("dtype,d,B", [("bf16", 128, 128), ("f32", 64, 64)])
def test_pool_and_attention_on_chunked_blocks(dtype, d, B):
    wl, pp, blen = chunked_case(d=d, dtype=dtype, B=B, zext=(3, 9, 16) if B == 128 else (5, 4, 8),
                                N_grid=(6, 18, 32) if B == 128 else (5, 8, 16))
    hs = range(wl.heads)
    Q, K, V = (np.stack(synth.gen_heads(wl, t, hs), axis=1) for t in (synth.Q_ID, synth.K_ID, synth.V_ID))
    np_, nb = pp.size, blen.size
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    q, k, v = (torch.from_numpy(x).to(dev).to(tdt) for x in (Q, K, V))
    qb, kb, vb = (torch.full((np_, wl.heads, d), 9.0, dtype=tdt, device=dev) for _ in range(3))
    qbar = torch.empty(wl.heads, nb, d, device=dev)
    kbar = torch.empty_like(qbar)
    dpp = torch.from_numpy(pp.astype(np.int32)).to(dev)
    P.prism_pool_score_chunked(q, k, v, dpp, B, qb, kb, vb, qbar, kbar)
    assert P.status_check() == 0
    valid = pp >= 0
    Qp = np.zeros((np_, wl.heads, d))
    Qp[valid] = Q[pp[valid]]
    assert np.array_equal(qb.float().cpu().numpy(), Qp)  # gathered rows exact, padding rows zero
    np.testing.assert_allclose(qbar.cpu().numpy(), po.block_mean(Qp, B, blen), atol=2e-6, rtol=1e-5)
    # attention over random kept lists of the chunked blocks
    counts, idx = synth.gen_block_lists(nb, wl.heads, seed=nb)
    Kp, Vp = np.zeros_like(Qp), np.zeros_like(Qp)
    Kp[valid], Vp[valid] = K[pp[valid]], V[pp[valid]]
    c, ix, bl = (torch.from_numpy(a.astype(np.int32)).to(dev) for a in (counts, idx, blen))
    o = torch.empty_like(qb)
    lse = torch.empty(wl.heads, np_, device=dev)
    P.prism_bsa_fwd(qb, kb, vb, B, c, ix, o, lse, blen=bl)
    assert P.status_check() == 0
    O, L = po.bsa_forward(Qp, Kp, Vp, counts, idx, B, blen=blen)
    tol = dict(max_abs=2e-2, mean_abs=2e-3) if dtype == "bf16" else dict(max_abs=2e-4, mean_abs=2e-5)
    attn_close(o.float().cpu().numpy()[valid], O[valid], what="O", **tol)
    np.testing.assert_allclose(lse.cpu().numpy()[:, valid], L[:, valid], atol=2e-3 if dtype == "bf16" else 1e-4)
    # backward from the oracle's O and lse; padding rows of dO hold noise the library must ignore
    dO = np.random.default_rng(2).normal(size=Qp.shape).astype(np.float32)
    O_in = synth.round_inputs(wl, np.nan_to_num(O).astype(np.float32))
    L_in = np.nan_to_num(L, nan=0.0).astype(np.float32)
    dO = synth.round_inputs(wl, dO)
    dQ, dK, dV = po.bsa_backward(Qp, Kp, Vp, O_in.astype(np.float64), dO.astype(np.float64),
                                 L_in.astype(np.float64), counts, idx, B, blen=blen)
    o_in, do_in = (torch.from_numpy(x).to(dev).to(tdt) for x in (O_in, dO))
    dq, dk, dv = (torch.full_like(qb, float("nan")) for _ in range(3))
    P.prism_bsa_bwd(qb, kb, vb, o_in, do_in, torch.from_numpy(L_in).to(dev), B, c, ix, dq, dk, dv, blen=bl)
    assert P.status_check() == 0
    for got, ref, name in ((dq, dQ, "dQ"), (dk, dK, "dK"), (dv, dV, "dV")):
        attn_close(got.float().cpu().numpy()[valid], ref[valid], what=name, **tol)


def test_tiny_layer_on_chunked_blocks():
    wl = synth.WORKLOADS["tiny"]
    layer = PrismLayer(wl, dev, train=False, chunked=True)
    layer.load_inputs()
    layer.forward()
    assert P.status_check() == 0
    hs = range(wl.heads)
    Q, K, V = (np.stack(synth.gen_heads(wl, t, hs), axis=1).astype(np.float64)
               for t in (synth.Q_ID, synth.K_ID, synth.V_ID))
    zs, _, _ = po.zone_shapes([V.reshape(wl.N, -1)], synth.gen_a2v(wl), wl.grid, wl.zone, wl.shapes)
    assert np.array_equal(layer.zone_shape.cpu().numpy(), zs)
    pp, blen = po.block_permutation_chunked(wl.grid, wl.zone, zs, wl.shapes, wl.block)
    assert np.array_equal(layer.perm_padded.cpu().numpy(), pp) and np.array_equal(layer.blen.cpu().numpy(), blen)
    valid = pp >= 0
    Qp, Kp, Vp = (np.zeros((pp.size, wl.heads, wl.d)) for _ in range(3))
    Qp[valid], Kp[valid], Vp[valid] = Q[pp[valid]], K[pp[valid]], V[pp[valid]]
    S = po.block_scores(po.block_mean(Qp, wl.block, blen), po.block_mean(Kp, wl.block, blen))
    stats, _ = check_lists(layer.counts.cpu().numpy(), layer.idx.cpu().numpy(), S, wl.sparsity, wl.cdf_tau)
    assert stats["exact"] == stats["rows"], stats
    counts, idx = po.select(S, wl.sparsity, wl.cdf_tau)
    O, _ = po.bsa_forward(Qp, Kp, Vp, counts, idx, wl.block, blen=blen)
    attn_close(layer.o_blk.double().cpu().numpy()[valid], O[valid], max_abs=2e-4, mean_abs=2e-5, what="O")
