"""A Prism attention layer with its heads split over the ranks of a process group.

One process per GPU.  Attention is independent per head, so pool + score, selection,
the forward and the backward of a rank's own heads need nothing from the other ranks.
The zone step is the one place where heads meet: it reads V's channels of every head.
Its statistic is a sum over channels (the per-axis line variance of each channel,
averaged), so every rank computes the partial sums of its own heads' channels
(prism_zone_partials), the ranks all-gather those [Z, 3] arrays, and every rank sums
them in rank order (prism_zone_shapes_from_partials): all ranks get the same zone
shapes and permutation, in every run.

Sequence-parallel training (the Prism page, "Data preparation and training procedure",
trains with FSDP and sequence parallelism) holds activations as token slices of all
heads.  `to_heads` / `to_tokens` are the all-to-all exchanges (Ulysses style) that turn
such a slice into all tokens of this rank's heads and back; the layer runs in between.

No kernel reads another GPU's memory: the only exchanges are the collectives here, on
whole tensors, between library calls.  `ops` is the per-rank compute; by default the
library's calls on this rank's CUDA device.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from . import prism as P


def head_range(heads: int, rank: int, world: int):
    """Heads [h0, h1) of `rank` when `heads` are split as evenly as possible over `world`."""
    return heads * rank // world, heads * (rank + 1) // world


def token_range(n: int, rank: int, world: int):
    """Tokens [t0, t1) of `rank` in a sequence-parallel split of n tokens."""
    return n * rank // world, n * (rank + 1) // world


class LibraryOps:
    """The per-rank compute of a sharded layer: the library's calls (CUDA tensors)."""

    def __init__(self):
        self.ws = {}

    def zone_partials(self, feat, C, grid, zone):
        T, H, W = grid
        Z = -(-T // zone[0]) * -(-H // zone[1]) * -(-W // zone[2])
        out = torch.empty(Z, 3, dtype=torch.float32, device=feat.device)
        self.ws["zp"] = P.prism_zone_partials(feat, C, grid, zone, out, self.ws.get("zp"))
        return out

    def zone_from_partials(self, parts, C_total, a2v, grid, zone, shapes):
        Z = parts.shape[1]
        zs = torch.empty(Z, dtype=torch.int32, device=parts.device)
        perm = torch.empty(a2v.numel(), dtype=torch.int32, device=parts.device)
        self.ws["zf"] = P.prism_zone_shapes_from_partials(parts, C_total, a2v, grid, zone, shapes, zs, perm,
                                                          self.ws.get("zf"))
        return zs, perm

    def pool_score_select(self, q, k, v, perm, B, sparsity, tau):
        N, Hh, d = q.shape
        nb = -(-N // B)
        q_blk, k_blk, v_blk = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        qbar = torch.empty(Hh, nb, d, dtype=torch.float32, device=q.device)
        kbar = torch.empty_like(qbar)
        scores = torch.empty(Hh, nb, nb, dtype=torch.float32, device=q.device)
        P.prism_pool_score(q, k, v, perm, B, q_blk, k_blk, v_blk, qbar, kbar, scores)
        counts = torch.empty(Hh, nb, dtype=torch.int32, device=q.device)
        idx = torch.empty(Hh, nb, nb, dtype=torch.int32, device=q.device)
        P.prism_select(scores, sparsity, tau, counts, idx)
        return q_blk, k_blk, v_blk, counts, idx

    def forward(self, q_blk, k_blk, v_blk, B, counts, idx):
        N, Hh, _ = q_blk.shape
        o = torch.empty_like(q_blk)
        lse = torch.empty(Hh, N, dtype=torch.float32, device=q_blk.device)
        self.ws["f"] = P.prism_bsa_fwd(q_blk, k_blk, v_blk, B, counts, idx, o, lse, self.ws.get("f"))
        return o, lse

    def backward(self, q_blk, k_blk, v_blk, o, do, lse, B, counts, idx):
        dq, dk, dv = (torch.empty_like(q_blk) for _ in range(3))
        self.ws["b"] = P.prism_bsa_bwd(q_blk, k_blk, v_blk, o, do, lse, B, counts, idx, dq, dk, dv,
                                       self.ws.get("b"))
        return dq, dk, dv


class HeadShardedLayer:
    """One attention layer of a workload, this rank's heads [h0, h1) of it.

    Inputs are this rank's heads of Q, K, V (and dO) as [N, Hh_local, d] tensors in
    raster order (dO in block order), and the whole A2V field [N]; outputs are this
    rank's heads of O (block order) and, when training, dQ, dK, dV (block order)."""

    def __init__(self, wl, group=None, ops=None, sparsity=None):
        self.wl = wl
        self.group = group
        self.rank = dist.get_rank(group) if dist.is_initialized() else 0
        self.world = dist.get_world_size(group) if dist.is_initialized() else 1
        self.h0, self.h1 = head_range(wl.heads, self.rank, self.world)
        self.ops = ops if ops is not None else LibraryOps()
        self.sparsity = wl.sparsity if sparsity is None else sparsity

    def gather_partials(self, part):
        """[world, Z, 3]: every rank's partial sums, in rank order."""
        if self.world == 1:
            return part[None].contiguous()
        got = [torch.empty_like(part) for _ in range(self.world)]
        dist.all_gather(got, part.contiguous(), group=self.group)
        return torch.stack(got).contiguous()

    def zone_shapes(self, v, a2v):
        wl = self.wl
        C_local = (self.h1 - self.h0) * wl.d
        if C_local == 0:  # more ranks than heads: this rank's channel slice is empty
            T, H, W = wl.grid
            Z = -(-T // wl.zone[0]) * -(-H // wl.zone[1]) * -(-W // wl.zone[2])
            part = torch.zeros(Z, 3, dtype=a2v.dtype, device=a2v.device)  # the partials' type
        else:
            part = self.ops.zone_partials(v.reshape(wl.N, C_local), C_local, wl.grid, wl.zone)
        parts = self.gather_partials(part)
        return self.ops.zone_from_partials(parts, wl.heads * wl.d, a2v, wl.grid, wl.zone, wl.shapes)

    def forward(self, q, k, v, a2v):
        """(zone_shape, perm, block-order Q/K/V, lists, O, lse) of this rank's heads."""
        wl = self.wl
        zs, perm = self.zone_shapes(v, a2v)
        if self.h1 == self.h0:
            self.saved = None
            return {"zone_shape": zs, "perm": perm}
        q_blk, k_blk, v_blk, counts, idx = self.ops.pool_score_select(q, k, v, perm, wl.block, self.sparsity,
                                                                      wl.cdf_tau)
        o, lse = self.ops.forward(q_blk, k_blk, v_blk, wl.block, counts, idx)
        self.saved = (q_blk, k_blk, v_blk, o, lse, counts, idx)
        return {"zone_shape": zs, "perm": perm, "counts": counts, "idx": idx, "o": o, "lse": lse}

    def backward(self, do):
        if self.saved is None:
            return None
        q_blk, k_blk, v_blk, o, lse, counts, idx = self.saved
        return self.ops.backward(q_blk, k_blk, v_blk, o, do, lse, self.wl.block, counts, idx)

    # ------------------------------------------------------- Ulysses exchanges
    def to_heads(self, x_tokens):
        """[n_local, Hh, d] (this rank's tokens, every head) -> [N, h1 - h0, d] (every
        token, this rank's heads): one all-to-all."""
        wl, W = self.wl, self.world
        n_loc = x_tokens.shape[0]
        hr = [head_range(wl.heads, r, W) for r in range(W)]
        send = torch.cat([x_tokens[:, a:b].reshape(-1) for a, b in hr])
        tr = [token_range(wl.N, r, W) for r in range(W)]
        hl = self.h1 - self.h0
        recv = torch.empty(wl.N * hl * wl.d, dtype=x_tokens.dtype, device=x_tokens.device)
        dist.all_to_all_single(recv, send, [(b - a) * hl * wl.d for a, b in tr],
                               [n_loc * (b - a) * wl.d for a, b in hr], group=self.group)
        return recv.view(wl.N, hl, wl.d)

    def to_tokens(self, x_heads):
        """Inverse of to_heads: [N, h1 - h0, d] -> [n_local, Hh, d]."""
        wl, W = self.wl, self.world
        t0, t1 = token_range(wl.N, self.rank, W)
        n_loc = t1 - t0
        tr = [token_range(wl.N, r, W) for r in range(W)]
        hr = [head_range(wl.heads, r, W) for r in range(W)]
        send = torch.cat([x_heads[a:b].reshape(-1) for a, b in tr])
        recv = torch.empty(n_loc * wl.heads * wl.d, dtype=x_heads.dtype, device=x_heads.device)
        dist.all_to_all_single(recv, send, [n_loc * (b - a) * wl.d for a, b in hr],
                               [(b - a) * (self.h1 - self.h0) * wl.d for a, b in tr], group=self.group)
        out = torch.empty(n_loc, wl.heads, wl.d, dtype=x_heads.dtype, device=x_heads.device)
        off = 0
        for a, b in hr:
            m = n_loc * (b - a) * wl.d
            out[:, a:b] = recv[off:off + m].view(n_loc, b - a, wl.d)
            off += m
        return out
