"""The head-sharded layer's host logic on 2 and 3 CPU ranks (gloo): head and token
ranges, the rank-ordered gather of the zone partial sums and the Ulysses exchanges.

The per-rank compute is the CPU oracle behind the layer's `ops` interface (test
infrastructure only; on a GPU the layer calls the library).  Gathered over ranks, the
sharded layer's zone shapes, permutation, kept lists, outputs and gradients must equal
the single-process oracle's on the tiny workload."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from audio_diffusion_dits_zone_b300 import sharded, synth
from oracle import prism_oracle as po


class OracleOps:
    """Per-rank compute of HeadShardedLayer on CPU tensors, from the oracle's functions."""

    def zone_partials(self, feat, C, grid, zone):
        v = po.zone_video_variation([feat.double().numpy()], grid, zone)  # sum_c mean-line variance / C
        ntok = np.array([(t1 - t0) * (h1 - h0) * (w1 - w0) for t0, t1, h0, h1, w0, w1 in po.zone_boxes(grid, zone)])
        return torch.from_numpy(v * C * ntok[:, None])

    def zone_from_partials(self, parts, C_total, a2v, grid, zone, shapes):
        ntok = np.array([(t1 - t0) * (h1 - h0) * (w1 - w0) for t0, t1, h0, h1, w0, w1 in po.zone_boxes(grid, zone)])
        total = np.zeros(parts.shape[1:])
        for p in parts.double().numpy():  # rank order
            total += p
        v = total / (C_total * ntok[:, None])
        u, abar = po.zone_a2v_coupling(a2v.double().numpy(), grid, zone)
        zs = po.choose_shapes(po.zone_axis_scores(v, u, abar), shapes)
        return torch.from_numpy(zs), torch.from_numpy(po.block_permutation(grid, zone, zs, shapes))

    def pool_score_select(self, q, k, v, perm, B, sparsity, tau):
        Q, K, V = (x.double().numpy() for x in (q, k, v))
        pm = perm.numpy()
        _, _, S = po.pool_score(Q, K, pm, B)
        counts, idx = po.select(S, sparsity, tau)
        return (torch.from_numpy(Q[pm]), torch.from_numpy(K[pm]), torch.from_numpy(V[pm]),
                torch.from_numpy(counts), torch.from_numpy(idx))

    def forward(self, q_blk, k_blk, v_blk, B, counts, idx):
        O, L = po.bsa_forward(q_blk.numpy(), k_blk.numpy(), v_blk.numpy(), counts.numpy(), idx.numpy(), B)
        return torch.from_numpy(O), torch.from_numpy(L)

    def backward(self, q_blk, k_blk, v_blk, o, do, lse, B, counts, idx):
        g = po.bsa_backward(q_blk.numpy(), k_blk.numpy(), v_blk.numpy(), o.numpy(), do.double().numpy(),
                            lse.numpy(), counts.numpy(), idx.numpy(), B)
        return tuple(torch.from_numpy(x) for x in g)


def inputs(wl):
    hs = range(wl.heads)
    q, k, v, do = (torch.from_numpy(np.stack(synth.gen_heads(wl, t, hs), axis=1)).double()
                   for t in (synth.Q_ID, synth.K_ID, synth.V_ID, synth.DO_ID))
    return q, k, v, do, torch.from_numpy(synth.gen_a2v(wl)).double()


def reference(wl):
    q, k, v, do, a2v = inputs(wl)
    ops = OracleOps()
    part = ops.zone_partials(v.reshape(wl.N, -1), wl.heads * wl.d, wl.grid, wl.zone)
    zs, perm = ops.zone_from_partials(part[None], wl.heads * wl.d, a2v, wl.grid, wl.zone, wl.shapes)
    qb, kb, vb, counts, idx = ops.pool_score_select(q, k, v, perm, wl.block, wl.sparsity, wl.cdf_tau)
    o, lse = ops.forward(qb, kb, vb, wl.block, counts, idx)
    return zs, perm, counts, idx, o, lse, ops.backward(qb, kb, vb, o, do, lse, wl.block, counts, idx)


def _run(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wl = synth.WORKLOADS["tiny"]
        q, k, v, do, a2v = inputs(wl)
        layer = sharded.HeadShardedLayer(wl, ops=OracleOps())
        h0, h1 = layer.h0, layer.h1
        # sequence-parallel inputs: this rank's tokens of every head, exchanged to heads
        t0, t1 = sharded.token_range(wl.N, rank, world)
        qh, kh, vh = (layer.to_heads(x[t0:t1].contiguous()) for x in (q, k, v))
        assert torch.equal(qh, q[:, h0:h1]) and torch.equal(vh, v[:, h0:h1])
        assert torch.equal(layer.to_tokens(qh), q[t0:t1])
        res = layer.forward(qh, kh, vh, a2v)
        grads = layer.backward(do[:, h0:h1]) if h1 > h0 else None
        zs, perm, counts, idx, o, lse, (dq, dk, dv) = reference(wl)
        assert torch.equal(res["zone_shape"], zs) and torch.equal(res["perm"], perm)
        if h1 > h0:
            assert torch.equal(res["counts"], counts[h0:h1]) and torch.equal(res["idx"], idx[h0:h1])
            np.testing.assert_allclose(res["o"].numpy(), o[:, h0:h1].numpy(), atol=1e-12)
            for g, r in zip(grads, (dq, dk, dv)):
                np.testing.assert_allclose(g.numpy(), r[:, h0:h1].numpy(), atol=1e-12)
        out[rank] = 1
    finally:
        dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("world", [2, 3])
def test_head_sharded_layer_equals_single_process(world):
    # world 3: uneven token split and a rank with no head of the 2-head workload
    out = mp.Manager().dict()
    mp.spawn(_run, args=(world, _free_port(), out), nprocs=world, join=True)
    assert sorted(out.keys()) == list(range(world))


def test_ranges_cover_without_overlap():
    for n, w in ((40, 8), (2, 3), (75600, 7)):
        hs = [sharded.head_range(n, r, w) for r in range(w)]
        assert hs[0][0] == 0 and hs[-1][1] == n and all(hs[i][1] == hs[i + 1][0] for i in range(w - 1))
        ts = [sharded.token_range(n, r, w) for r in range(w)]
        assert ts == hs
