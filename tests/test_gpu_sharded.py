"""The head-sharded layer's per-rank compute through the library, two ranks emulated in
one process on one GPU (the gather of the zone partials is a stack in rank order; no
kernel waits on another rank).  Each rank's results must equal the unsharded layer's
slice of heads: exactly for the zone step (up to fp32 near-ties of the shape costs),
the lists, the forward and dK / dV; within the bf16 tolerance for dQ, whose fp32
reduce-adds may sum in another order."""
import numpy as np
import pytest
import torch

from audio_diffusion_dits_zone_b300 import prism as P
from audio_diffusion_dits_zone_b300 import sharded, synth
from audio_diffusion_dits_zone_b300.pipeline import PrismLayer
from parity import attn_close, compare_perm_by_zone

pytestmark = pytest.mark.gpu


def test_two_rank_head_split_equals_unsharded_layer():
    wl = synth.Workload("shard", 80, (7, 20, 40), 4, 128, "bf16", (3, 9, 16), 128, synth.SHAPES_128, 0.8, 0.2, 2,
                        3.0, (44, 42, 42), "fwd+bwd")
    full = PrismLayer(wl, "cuda", train=True)
    full.load_inputs()
    full.step()
    assert P.status_check() == 0
    world = 2
    ops = sharded.LibraryOps()
    parts = []
    for r in range(world):
        h0, h1 = sharded.head_range(wl.heads, r, world)
        parts.append(ops.zone_partials(full.v[:, h0:h1].reshape(wl.N, (h1 - h0) * wl.d), (h1 - h0) * wl.d, wl.grid,
                                       wl.zone))
    zs, perm = ops.zone_from_partials(torch.stack(parts).contiguous(), wl.heads * wl.d, full.a2v, wl.grid, wl.zone,
                                      wl.shapes)
    assert P.status_check() == 0
    g, ref = zs.cpu().numpy(), full.zone_shape.cpu().numpy()
    assert (g != ref).sum() <= 1, (g, ref)  # fp32 sums of the channel halves in another grouping
    assert compare_perm_by_zone(perm.cpu().numpy(), full.perm.cpu().numpy(), g, ref, wl.grid, wl.zone) >= len(g) - 1
    if not np.array_equal(g, ref):
        pytest.skip("a zone shape sits on an fp32 near-tie; the per-head comparison needs the same permutation")
    for r in range(world):
        h0, h1 = sharded.head_range(wl.heads, r, world)
        qb, kb, vb, counts, idx = ops.pool_score_select(full.q[:, h0:h1], full.k[:, h0:h1], full.v[:, h0:h1], perm,
                                                        wl.block, wl.sparsity, wl.cdf_tau)
        assert torch.equal(counts, full.counts[h0:h1])
        for h in range(h1 - h0):
            for i in range(wl.nb):
                c = int(counts[h, i])
                assert torch.equal(idx[h, i, :c], full.idx[h0 + h, i, :c])
        o, lse = ops.forward(qb, kb, vb, wl.block, counts, idx)
        assert torch.equal(o, full.o_blk[:, h0:h1]) and torch.equal(lse, full.lse[h0:h1])
        dq, dk, dv = ops.backward(qb, kb, vb, o, full.do_blk[:, h0:h1].contiguous(), lse, wl.block, counts, idx)
        assert P.status_check() == 0
        assert torch.equal(dk, full.dk[:, h0:h1]) and torch.equal(dv, full.dv[:, h0:h1])
        attn_close(dq.float().cpu().numpy(), full.dq[:, h0:h1].float().cpu().numpy(), max_abs=2e-2, mean_abs=2e-4,
                   what=f"dQ rank {r}")
