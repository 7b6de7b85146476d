"""One Prism attention layer on the device: buffers for a workload and the calls of
the path in order (zone shapes -> pool + score -> select -> attention forward ->
backward).  PyTorch only provides the memory and the stream; every step is a
libprism call.
"""
from __future__ import annotations

import numpy as np
import torch

from . import prism as P
from . import synth


class PrismLayer:
    """Device-resident state of one attention layer for a ``synth.Workload``."""

    def __init__(self, wl: synth.Workload, device="cuda", sparsity=None, train=None, fused_select=False,
                 chunked=False):
        """fused_select: block scores and selection in one call (prism_score_select), the
        score matrix never written; otherwise prism_pool_score writes the scores and
        prism_select reads them.  chunked: zone-chunked blocks (every zone cut into B-token
        blocks of its own, in a padded block order with per-block lengths) instead of
        consecutive B-token chunks of the whole block order."""
        self.wl = wl
        self.fused_select = fused_select
        self.chunked = chunked
        self.device = torch.device(device)
        self.sparsity = wl.sparsity if sparsity is None else sparsity
        self.train = (wl.mode == "fwd+bwd") if train is None else train
        N, Hh, d, nb = wl.N, wl.heads, wl.d, wl.nb
        self.nrows = N  # rows of the block order (np for zone-chunked blocks)
        if chunked:
            nb, self.nrows = P.prism_zone_chunked_size(wl.grid, wl.zone, wl.block)
        self.nb = nb
        dt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
        self.dtype = dt
        e = dict(device=self.device)
        T, H, W = wl.grid
        self.Z = -(-T // wl.zone[0]) * -(-H // wl.zone[1]) * -(-W // wl.zone[2])
        self.q = torch.empty(N, Hh, d, dtype=dt, **e)
        self.k = torch.empty(N, Hh, d, dtype=dt, **e)
        self.v = torch.empty(N, Hh, d, dtype=dt, **e)
        self.a2v = torch.empty(N, dtype=torch.float32, **e)
        self.zone_shape = torch.empty(self.Z, dtype=torch.int32, **e)
        self.perm = torch.empty(N, dtype=torch.int32, **e)
        self.perm_padded = torch.empty(self.nrows, dtype=torch.int32, **e) if chunked else None
        self.blen = torch.empty(nb, dtype=torch.int32, **e) if chunked else None
        self.ws_chunk = None
        R = self.nrows
        self.q_blk = torch.empty(R, Hh, d, dtype=dt, **e)
        self.k_blk = torch.empty(R, Hh, d, dtype=dt, **e)
        self.v_blk = torch.empty(R, Hh, d, dtype=dt, **e)
        self.qbar = torch.empty(Hh, nb, d, dtype=torch.float32, **e)
        self.kbar = torch.empty(Hh, nb, d, dtype=torch.float32, **e)
        self.scores = None if fused_select else torch.empty(Hh, nb, nb, dtype=torch.float32, **e)
        self.counts = torch.empty(Hh, nb, dtype=torch.int32, **e)
        self.idx = torch.empty(Hh, nb, nb, dtype=torch.int32, **e)
        self.o_blk = torch.empty_like(self.q_blk)
        self.lse = torch.empty(Hh, R, dtype=torch.float32, **e)
        self.ws_zone = self.ws_fwd = self.ws_bwd = None
        if self.train:
            self.do_blk = torch.empty_like(self.q_blk)
            self.dq = torch.empty_like(self.q_blk)
            self.dk = torch.empty_like(self.q_blk)
            self.dv = torch.empty_like(self.q_blk)

    # ------------------------------------------------------------------ inputs
    def load_inputs(self, threads=8):
        """Generate the seeded inputs on the host and copy them into the device buffers."""
        wl = self.wl
        todo = [(synth.Q_ID, self.q), (synth.K_ID, self.k), (synth.V_ID, self.v)]
        if self.train:
            todo.append((synth.DO_ID, self.do_blk))
        for tensor, dst in todo:
            for h0 in range(0, wl.heads, 8):   # groups of heads bound the host memory
                heads = list(range(h0, min(h0 + 8, wl.heads)))
                rows = self.nrows if tensor == synth.DO_ID else 0
                for h, x in zip(heads, synth.gen_heads(wl, tensor, heads, threads, rows)):
                    dst[:, h, :].copy_(torch.from_numpy(x).to(self.dtype))
        self.a2v.copy_(torch.from_numpy(synth.gen_a2v(wl)))
        torch.cuda.synchronize(self.device)

    # ------------------------------------------------------------------- steps
    def zone_shapes(self, stream=None):
        wl = self.wl
        feat = self.v.view(wl.N, wl.heads * wl.d)
        self.ws_zone = P.prism_zone_shapes(feat, wl.heads * wl.d, self.a2v, wl.grid, wl.zone, wl.shapes,
                                           self.zone_shape, self.perm, self.ws_zone, stream)
        if self.chunked:
            self.ws_chunk = P.prism_zone_perm_chunked(self.zone_shape, wl.grid, wl.zone, wl.shapes, wl.block,
                                                      self.perm_padded, self.blen, self.ws_chunk, stream)

    def _pool(self, qbar, kbar, scores, stream):
        if self.chunked:
            P.prism_pool_score_chunked(self.q, self.k, self.v, self.perm_padded, self.wl.block, self.q_blk, self.k_blk,
                                       self.v_blk, qbar, kbar, scores, stream)
        else:
            P.prism_pool_score(self.q, self.k, self.v, self.perm, self.wl.block, self.q_blk, self.k_blk, self.v_blk,
                               qbar, kbar, scores, stream)

    def pool_score(self, stream=None):
        self._pool(self.qbar, self.kbar, self.scores, stream)

    def pool_copies(self, stream=None):
        """Block-order copies of Q, K, V with the current permutation only (no means, no
        scores): what a step that reuses an earlier step's selection needs."""
        self._pool(None, None, None, stream)

    def select(self, stream=None):
        if self.fused_select:
            P.prism_score_select(self.qbar, self.kbar, self.sparsity, self.wl.cdf_tau, self.counts, self.idx, stream)
        else:
            P.prism_select(self.scores, self.sparsity, self.wl.cdf_tau, self.counts, self.idx, stream)

    def _groups(self):
        g = self.wl.head_group or self.wl.heads
        return [(h0, min(h0 + g, self.wl.heads)) for h0 in range(0, self.wl.heads, g)]

    def attention_fwd(self, stream=None):
        B = self.wl.block
        for h0, h1 in self._groups():
            self.ws_fwd = P.prism_bsa_fwd(self.q_blk[:, h0:h1], self.k_blk[:, h0:h1], self.v_blk[:, h0:h1], B,
                                          self.counts[h0:h1], self.idx[h0:h1], self.o_blk[:, h0:h1],
                                          self.lse[h0:h1], self.ws_fwd, stream, blen=self.blen)

    def attention_bwd(self, stream=None):
        B = self.wl.block
        for h0, h1 in self._groups():
            self.ws_bwd = P.prism_bsa_bwd(self.q_blk[:, h0:h1], self.k_blk[:, h0:h1], self.v_blk[:, h0:h1],
                                          self.o_blk[:, h0:h1], self.do_blk[:, h0:h1], self.lse[h0:h1], B,
                                          self.counts[h0:h1], self.idx[h0:h1], self.dq[:, h0:h1],
                                          self.dk[:, h0:h1], self.dv[:, h0:h1], self.ws_bwd, stream, blen=self.blen)

    def forward(self, stream=None):
        self.zone_shapes(stream)
        self.pool_score(stream)
        self.select(stream)
        self.attention_fwd(stream)

    def step(self, stream=None):
        """One pass of the whole path: forward, plus backward when training."""
        self.forward(stream)
        if self.train:
            self.attention_bwd(stream)

    # ------------------------------------------------------------------- work
    def block_lengths(self):
        """Tokens of every block (int64 device tensor)."""
        wl = self.wl
        if self.chunked:
            return self.blen.long()
        lens = torch.full((wl.nb,), wl.block, dtype=torch.int64, device=self.device)
        lens[-1] = wl.N - wl.block * (wl.nb - 1)
        return lens

    def executed_pairs(self) -> np.ndarray:
        """Per (head, query block): sum over kept blocks of |b_i| * |b_j| (token pairs)."""
        lens = self.block_lengths()
        nbr = torch.arange(self.nb, device=self.device)
        valid = nbr[None, None, :] < self.counts[:, :, None].long()
        jl = lens[self.idx.long().clamp(0, self.nb - 1)] * valid
        return (jl.sum(-1) * lens[None, :]).cpu().numpy()

    def flops(self):
        """(executed fwd FLOPs, executed bwd FLOPs, dense-equivalent fwd, dense bwd)."""
        wl = self.wl
        pairs = float(self.executed_pairs().sum())
        dense = float(wl.N) * wl.N * wl.heads
        return 4.0 * pairs * wl.d, 10.0 * pairs * wl.d, 4.0 * dense * wl.d, 10.0 * dense * wl.d
