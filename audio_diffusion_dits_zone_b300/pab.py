"""Attention broadcast across diffusion steps for the Prism layer.

"Real-time video generation with pyramid attention broadcast" (method and results):
over the steps of a diffusion sampler the difference between consecutive steps'
attention outputs is U-shaped, small through the middle ~70% of the steps; there an
attention's output can be computed once and broadcast (reused) for the next few steps,
each attention with its own broadcast range, chosen from the mean squared error between
consecutive steps' outputs (spatial attention, the most variable, gets the widest range).

Applied to the Prism layer (readings where the page is silent):
  * the broadcast window is steps [round(0.15 T), round(0.85 T)); inside it attention
    is computed at the window's first step and every (range + 1) steps after, each
    computed output serving the `range` steps that follow; outside it every step
    computes;
  * mode "outputs" reuses the computed attention output itself (the step runs no
    kernel); mode "lists" reuses only Prism's selection of that step (zone shapes,
    permutation, kept lists) and recomputes attention with the step's own Q, K, V, so
    the selection's cost is what is broadcast;
  * `calibrate` runs a trajectory with the selection fixed (every step computing
    attention with the first step's lists, so the outputs share one permutation) and
    returns the per-head MSE between consecutive steps (prism_attn_mse): the curve the
    broadcast range is read from.
"""
from __future__ import annotations

import torch

from . import prism as P


def schedule(n_steps: int, broadcast_range: int, window=(0.15, 0.85)) -> list:
    """Per step: True where attention is computed, False where it is broadcast."""
    lo, hi = int(round(window[0] * n_steps)), int(round(window[1] * n_steps))
    return [not (lo <= t < hi) or (t - lo) % (broadcast_range + 1) == 0 for t in range(n_steps)]


class BroadcastLayer:
    """A PrismLayer driven through the steps of a denoising trajectory with attention
    broadcast.  Before run_step(t) the caller writes step t's inputs into layer.q,
    layer.k, layer.v (raster order) and layer.a2v; after it, layer.o_blk holds the
    step's attention output in the block order of layer.perm."""

    def __init__(self, layer, n_steps: int, broadcast_range: int, mode: str = "outputs"):
        assert mode in ("outputs", "lists")
        self.layer = layer
        self.plan = schedule(n_steps, broadcast_range)
        self.mode = mode

    def run_step(self, t: int, stream=None) -> bool:
        """Run step t; returns whether attention was computed in full (selection included)."""
        L = self.layer
        if self.plan[t]:
            L.forward(stream)
            return True
        if self.mode == "lists":
            L.pool_copies(stream)
            L.attention_fwd(stream)
        return False


def calibrate(layer, set_step_inputs, n_steps: int, stream=None):
    """[n_steps - 1, Hh] fp32 MSE between consecutive steps' attention outputs, with the
    selection of step 0 held for the whole trajectory.  set_step_inputs(t) writes step
    t's inputs into the layer."""
    set_step_inputs(0)
    layer.forward(stream)
    prev = layer.o_blk.clone()
    out = torch.empty(n_steps - 1, layer.wl.heads, dtype=torch.float32, device=layer.device)
    ws = None
    for t in range(1, n_steps):
        set_step_inputs(t)
        layer.pool_copies(stream)
        layer.attention_fwd(stream)
        ws = P.prism_attn_mse(layer.o_blk, prev, out[t - 1], ws, stream)
        prev.copy_(layer.o_blk)
    return out
