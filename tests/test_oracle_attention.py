"""Pins for the oracle's block-sparse attention forward and backward.

Sparsity 0 must equal dense softmax attention; any kept lists must equal an
explicit token mask fed to torch's scaled_dot_product_attention (a library
routine) in fp64, forward and, through torch.autograd, backward.  Identical
keys give the mean of the kept values.
"""
import math

import numpy as np
import pytest
import torch

from oracle import prism_oracle as po
from audio_diffusion_dits_zone_b300 import synth


def token_mask(counts, idx, N, B):
    Hh, nb = counts.shape
    M = np.zeros((Hh, N, N), dtype=bool)
    for h in range(Hh):
        for i in range(nb):
            cols = po.kept_tokens(idx[h, i, : counts[h, i]], B, N)
            M[h, i * B:min((i + 1) * B, N)][:, cols] = True
    return M


def sdpa(Q, K, V, mask=None):
    """torch SDPA in fp64 over heads: inputs [N, Hh, d] -> [N, Hh, d]."""
    q, k, v = (torch.as_tensor(x).permute(1, 0, 2)[None] for x in (Q, K, V))
    m = None if mask is None else torch.as_tensor(mask)[None]
    return torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=m)[0].permute(1, 0, 2)


def rand_qkv(N, Hh, d, seed):
    rng = np.random.default_rng(seed)
    return [rng.normal(size=(N, Hh, d)) for _ in range(3)]


@pytest.mark.parametrize("N,B", [(64, 16), (70, 16)])
def test_sparsity_zero_is_dense_attention(N, B):
    Hh, d = 2, 32
    Q, K, V = rand_qkv(N, Hh, d, 0)
    nb = -(-N // B)
    counts = np.full((Hh, nb), nb, np.int32)
    idx = np.broadcast_to(np.arange(nb, dtype=np.int32), (Hh, nb, nb)).copy()
    O, LSE = po.bsa_forward(Q, K, V, counts, idx, B)
    np.testing.assert_allclose(O, sdpa(Q, K, V).numpy(), rtol=1e-10, atol=1e-12)
    S = np.einsum("nhd,mhd->hnm", Q, K) / math.sqrt(d)
    np.testing.assert_allclose(LSE, np.log(np.exp(S).sum(-1)), rtol=1e-12)


@pytest.mark.parametrize("N,B,seed", [(96, 16, 1), (100, 16, 2), (64, 64, 3)])
def test_masked_forward_and_backward_match_sdpa(N, B, seed):
    Hh, d = 2, 16
    Q, K, V = rand_qkv(N, Hh, d, seed)
    nb = -(-N // B)
    counts, idx = synth.gen_block_lists(nb, Hh, seed=seed)
    O, LSE = po.bsa_forward(Q, K, V, counts, idx, B)
    mask = token_mask(counts, idx, N, B)
    q, k, v = (torch.tensor(x, requires_grad=True) for x in (Q, K, V))
    ref = sdpa(q, k, v, mask)
    np.testing.assert_allclose(O, ref.detach().numpy(), rtol=1e-10, atol=1e-12)
    dO = np.random.default_rng(seed + 10).normal(size=(N, Hh, d))
    ref.backward(torch.tensor(dO))
    dQ, dK, dV = po.bsa_backward(Q, K, V, O, dO, LSE, counts, idx, B)
    np.testing.assert_allclose(dQ, q.grad.numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(dK, k.grad.numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(dV, v.grad.numpy(), rtol=1e-9, atol=1e-11)


def test_identical_keys_average_kept_values():
    N, Hh, d, B = 48, 1, 8, 16
    rng = np.random.default_rng(4)
    Q = rng.normal(size=(N, Hh, d))
    K = np.broadcast_to(rng.normal(size=(1, Hh, d)), (N, Hh, d)).copy()
    V = rng.normal(size=(N, Hh, d))
    counts = np.array([[1, 2, 3]], np.int32)
    idx = np.array([[[2, -1, -1], [0, 2, -1], [0, 1, 2]]], np.int32)
    O, _ = po.bsa_forward(Q, K, V, counts, idx, B)
    np.testing.assert_allclose(O[0:16, 0], np.broadcast_to(V[32:48, 0].mean(0), (16, d)))
    np.testing.assert_allclose(O[16:32, 0], np.broadcast_to(np.r_[V[0:16, 0], V[32:48, 0]].mean(0), (16, d)))
    np.testing.assert_allclose(O[32:48, 0], np.broadcast_to(V[:, 0].mean(0), (16, d)))


def test_empty_list_gives_zero_output():
    N, Hh, d, B = 32, 1, 4, 16
    Q, K, V = rand_qkv(N, Hh, d, 5)
    counts = np.array([[0, 2]], np.int32)
    idx = np.array([[[-1, -1], [0, 1]]], np.int32)
    O, LSE = po.bsa_forward(Q, K, V, counts, idx, B)
    assert np.all(O[:16] == 0) and np.all(np.isneginf(LSE[0, :16]))
    dQ, dK, dV = po.bsa_backward(Q, K, V, O, np.ones_like(Q), LSE, counts, idx, B)
    assert np.all(dQ[:16] == 0)


def test_sampled_backward_equals_full_backward():
    N, Hh, d, B = 112, 2, 16, 16
    Q, K, V = rand_qkv(N, Hh, d, 6)
    nb = -(-N // B)
    counts, idx = synth.gen_block_lists(nb, Hh, seed=6)
    dO = np.random.default_rng(7).normal(size=(N, Hh, d))
    O, LSE = po.bsa_forward(Q, K, V, counts, idx, B)
    dQ, dK, dV = po.bsa_backward(Q, K, V, O, dO, LSE, counts, idx, B)
    dq, dk, dv = po.bsa_backward_sampled(Q, K, V, dO, counts, idx, B, 1, [0, 6], [3, 6])
    for i in (0, 6):
        np.testing.assert_allclose(dq[i], dQ[i * B:min((i + 1) * B, N), 1], rtol=1e-10, atol=1e-12)
    for j in (3, 6):
        np.testing.assert_allclose(dk[j], dK[j * B:min((j + 1) * B, N), 1], rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(dv[j], dV[j * B:min((j + 1) * B, N), 1], rtol=1e-10, atol=1e-12)


def test_chain_on_tiny_workload_runs_and_is_sane():
    wl = synth.WORKLOADS["tiny"]
    heads = range(wl.heads)
    Q = np.stack(synth.gen_heads(wl, synth.Q_ID, heads), axis=1)
    K = np.stack(synth.gen_heads(wl, synth.K_ID, heads), axis=1)
    V = np.stack(synth.gen_heads(wl, synth.V_ID, heads), axis=1)
    a2v = synth.gen_a2v(wl)
    zs, perm, det = po.zone_shapes([V.reshape(wl.N, -1)], a2v, wl.grid, wl.zone, wl.shapes)
    assert zs.shape == (4,) and np.array_equal(np.sort(perm), np.arange(wl.N))
    qbar, kbar, S = po.pool_score(Q, K, perm, wl.block)
    counts, idx = po.select(S, wl.sparsity, wl.cdf_tau)
    assert counts.shape == (wl.heads, wl.nb) and np.all(counts >= 3)
    O, LSE = po.bsa_forward(Q[perm], K[perm], V[perm], counts, idx, wl.block)
    assert np.isfinite(O).all() and np.isfinite(LSE).all()
