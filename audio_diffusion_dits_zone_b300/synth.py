"""Seeded synthetic inputs shaped like Wan-VAE video latents at 720p / 1080p / 2K.

This module only *draws inputs*.  It holds none of the arithmetic of the method
(zones, pooling, selection, attention): both the CUDA path and the CPU oracle
receive their inputs from here and from nowhere else, so that neither has to
trust the other for what it is fed.

Workload shapes (Prism page, "Data preparation and training procedure" and
"Resolution and hardware requirements"): clips are encoded to Wan-VAE latents,
frame counts have the form 4k+1, resolutions are 720p / 1080p / 2K.  81 video
frames become T = 1 + 80/4 = 21 latent frames; a 1280x720 frame becomes an 80x45
token grid after the VAE's 8x and the patchifier's 2x reduction (1920x1080 ->
120x68, 2560x1440 -> 160x90).

Input recipe (the pages fix none of it; these are the readings used here):
  * Q, K, V per (tensor, head): x[p,:] = sum_{m<6} a_m sin(2 pi f_m . p + phi_m)
    + eps, with p = (t,h,w) token coordinates, f_m ~ U[0,0.25)^3 cycles/token,
    phi_m ~ U[0, 2 pi), a_m ~ N(0, 1/6) per channel (variance 1/6), eps ~ N(0, 0.1^2).
  * 3D rotary position embedding (theta = 10000, adjacent channel pairs) on Q and
    K only, channels split t:h:w = 16:24:24 (d=64) or 44:42:42 (d=128).  V keeps
    the content unrotated, as attention values do.
  * A2V cross-attention feature-norm field: a sum of unit-amplitude isotropic 3D
    Gaussian bumps over token coordinates, centres uniform over the grid.
  * dO ~ N(0, 1) per (head), in block order (it is i.i.d., so the order is moot).
  * Audio-to-video cross-attention (the step that produces the A2V field): video
    queries drawn like V (sinusoids over (t,h,w) + noise, no rotary embedding, since
    audio and video share no position frame); audio keys and values per head the
    same way over the 1D audio time axis (6 sinusoids of frequency U[0, 0.25)
    cycles/token + noise).  AUDIO_TOKENS = 157 audio tokens: the 81 video frames at
    16 fps span 5.06 s, taken at 31 audio latent frames per second (a reading; the
    pages give no audio token rate).
  * Denoising trajectory (attention broadcast across diffusion steps): step t of n
    takes x_t = (1 - sigma_t) x + sigma_t e with sigma_t = 1 - t / (n - 1) (a linear
    rectified-flow path), x the workload's Q, K or V and e ~ N(0, 1) per (tensor, head).
  * Seeds: numpy PCG64 from SeedSequence([0, config id, tensor id, head]).

Values are generated in float32; ``to_bf16`` rounds them to bfloat16 (round to
nearest even) for the configurations that run in bf16.  Both sides round with
the same function, on the host, before anything else touches the data.
"""
from __future__ import annotations

import math
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

Q_ID, K_ID, V_ID, DO_ID = 0, 1, 2, 3
A2V_ID = 100
AQ_ID, AK_ID, AV_ID = 10, 11, 12  # video queries, audio keys, audio values of the cross-attention
AUDIO_TOKENS = 157


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: grid, heads, blocks, zones and selection settings."""

    name: str
    cid: int                      # config id used in the seeds
    grid: tuple                   # (T, H, W) latent token grid
    heads: int
    d: int
    dtype: str                    # "f32" or "bf16"
    zone: tuple                   # macro-zone extents (Zt, Zh, Zw)
    block: int                    # tokens per block B
    shapes: tuple                 # block-shape set ((et, eh, ew), ...)
    sparsity: float
    cdf_tau: float
    bumps: int
    sigma: float
    rope_split: tuple             # channels per axis (t, h, w)
    mode: str                     # "fwd" or "fwd+bwd"
    head_group: int = 0           # heads per attention launch (0 = all heads)
    sweep: tuple = field(default=())

    @property
    def N(self) -> int:
        T, H, W = self.grid
        return T * H * W

    @property
    def nb(self) -> int:
        return -(-self.N // self.block)


SHAPES_128 = ((1, 8, 16), (2, 8, 8), (4, 4, 8), (8, 4, 4))
SHAPES_64 = ((1, 8, 8), (2, 4, 8), (4, 4, 4), (8, 2, 4))

WORKLOADS = {
    "tiny": Workload("tiny", 0, (5, 8, 16), 2, 64, "f32", (5, 4, 8), 64, SHAPES_64,
                     0.75, 0.20, 1, 3.0, (16, 24, 24), "fwd+bwd"),
    "720p": Workload("720p", 1, (21, 45, 80), 40, 128, "bf16", (3, 9, 16), 128, SHAPES_128,
                     0.80, 0.20, 1, 3.0, (44, 42, 42), "fwd"),
    "1080p": Workload("1080p", 2, (21, 68, 120), 40, 128, "bf16", (3, 9, 16), 128, SHAPES_128,
                      0.85, 0.20, 2, 3.0, (44, 42, 42), "fwd"),
    "2k": Workload("2k", 3, (21, 90, 160), 40, 128, "bf16", (3, 9, 16), 128, SHAPES_128,
                   0.93, 0.20, 3, 6.0, (44, 42, 42), "fwd", head_group=8),
    "train720p": Workload("train720p", 4, (21, 45, 80), 40, 128, "bf16", (3, 9, 16), 128,
                          SHAPES_128, 0.80, 0.20, 1, 3.0, (44, 42, 42), "fwd+bwd",
                          sweep=(0.0, 0.75, 0.80, 0.85, 0.93)),
    # the 720p training layer with 4 heads: a small case of the same kernels for profiling
    "720p-4h": Workload("720p-4h", 5, (21, 45, 80), 4, 128, "bf16", (3, 9, 16), 128, SHAPES_128,
                        0.80, 0.20, 1, 3.0, (44, 42, 42), "fwd+bwd"),
    # the 2K forward layer with 4 heads (2,363 blocks per row): the profiling case of the
    # selection kernels at that row length
    "2k-4h": Workload("2k-4h", 6, (21, 90, 160), 4, 128, "bf16", (3, 9, 16), 128, SHAPES_128,
                      0.93, 0.20, 3, 6.0, (44, 42, 42), "fwd"),
}


def _rng(*key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([0, *key])))


def _coords(grid):
    T, H, W = grid
    t = np.arange(T, dtype=np.float64)[:, None, None]
    h = np.arange(H, dtype=np.float64)[None, :, None]
    w = np.arange(W, dtype=np.float64)[None, None, :]
    return t, h, w


def rope_tables(grid, d: int, split: tuple, theta: float = 10000.0):
    """cos/sin tables [N, d/2] for a 3D rotary embedding on adjacent channel pairs.

    Channel pairs are assigned to the t, h and w axes in that order, ``split``
    channels each; pair k of an axis group of g channels turns by
    pos_axis * theta^(-2k/g).
    """
    T, H, W = grid
    assert sum(split) == d and all(s % 2 == 0 for s in split)
    t, h, w = _coords(grid)
    pos = [np.broadcast_to(a, (T, H, W)).reshape(-1) for a in (t, h, w)]
    angles = []
    for axis, g in enumerate(split):
        k = np.arange(g // 2, dtype=np.float64)
        inv = theta ** (-2.0 * k / g)
        angles.append(pos[axis][:, None] * inv[None, :])
    ang = np.concatenate(angles, axis=1)
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


def _apply_rope(x: np.ndarray, cos: np.ndarray, sin: np.ndarray) -> np.ndarray:
    x0 = x[:, 0::2]
    x1 = x[:, 1::2]
    out = np.empty_like(x)
    out[:, 0::2] = x0 * cos - x1 * sin
    out[:, 1::2] = x0 * sin + x1 * cos
    return out


def gen_head(wl: Workload, tensor: int, head: int, rope=None) -> np.ndarray:
    """One head of Q (tensor 0), K (1) or V (2) in raster token order: float32 [N, d]."""
    rng = _rng(wl.cid, tensor, head)
    f = rng.uniform(0.0, 0.25, size=(6, 3))
    phi = rng.uniform(0.0, 2.0 * math.pi, size=6)
    a = rng.normal(0.0, math.sqrt(1.0 / 6.0), size=(6, wl.d))
    t, h, w = _coords(wl.grid)
    waves = np.empty((wl.N, 6), dtype=np.float64)
    for m in range(6):
        ph = 2.0 * math.pi * (f[m, 0] * t + f[m, 1] * h + f[m, 2] * w) + phi[m]
        waves[:, m] = np.sin(ph).reshape(-1)
    x = (waves @ a).astype(np.float32)
    x += rng.standard_normal((wl.N, wl.d), dtype=np.float32) * np.float32(0.1)
    if tensor in (Q_ID, K_ID):
        cos, sin = rope if rope is not None else rope_tables(wl.grid, wl.d, wl.rope_split)
        x = _apply_rope(x, cos, sin)
    return x


def gen_audio_head(wl: Workload, tensor: int, head: int, M: int = AUDIO_TOKENS) -> np.ndarray:
    """One head of the audio keys (AK_ID) or values (AV_ID): float32 [M, d] over the
    audio time axis."""
    rng = _rng(wl.cid, tensor, head)
    f = rng.uniform(0.0, 0.25, size=6)
    phi = rng.uniform(0.0, 2.0 * math.pi, size=6)
    a = rng.normal(0.0, math.sqrt(1.0 / 6.0), size=(6, wl.d))
    tau = np.arange(M, dtype=np.float64)[:, None]
    waves = np.sin(2.0 * math.pi * f[None, :] * tau + phi[None, :])
    x = (waves @ a).astype(np.float32)
    x += rng.standard_normal((M, wl.d), dtype=np.float32) * np.float32(0.1)
    return x


def gen_a2v_inputs(wl: Workload, heads, M: int = AUDIO_TOKENS):
    """Video queries [N, Hh, d] and audio keys / values [M, Hh, d] of the cross-attention,
    rounded like every other input of the workload."""
    heads = list(heads)
    with ThreadPoolExecutor(max_workers=8) as ex:
        qv = np.stack(list(ex.map(lambda h: round_inputs(wl, gen_head(wl, AQ_ID, h)), heads)), axis=1)
    ka = np.stack([round_inputs(wl, gen_audio_head(wl, AK_ID, h, M)) for h in heads], axis=1)
    va = np.stack([round_inputs(wl, gen_audio_head(wl, AV_ID, h, M)) for h in heads], axis=1)
    return qv, ka, va


NOISE_ID = 20  # + tensor id: the noise end of a denoising trajectory


def trajectory_sigma(t: int, n_steps: int) -> float:
    """Noise level of step t of an n-step denoising trajectory: 1 at the first step,
    linearly down to 0 at the last (a rectified-flow path, as Wan's sampler takes)."""
    return 1.0 - t / max(1, n_steps - 1)


def gen_noise_head(wl: Workload, tensor: int, head: int) -> np.ndarray:
    """One head of the trajectory's noise for tensor Q, K or V: float32 [N, d] ~ N(0, 1)."""
    return _rng(wl.cid, NOISE_ID + tensor, head).standard_normal((wl.N, wl.d), dtype=np.float32)


def gen_noise_heads(wl: Workload, tensor: int, heads, threads: int = 8) -> list:
    """Several heads of the trajectory noise of one tensor, in parallel threads."""
    with ThreadPoolExecutor(max_workers=threads) as ex:
        return list(ex.map(lambda h: gen_noise_head(wl, tensor, h), list(heads)))


def trajectory_blend(clean: np.ndarray, noise: np.ndarray, t: int, n_steps: int) -> np.ndarray:
    """Input of step t: (1 - sigma) * clean + sigma * noise in float32, rounded like the
    workload's inputs by the caller."""
    sg = np.float32(trajectory_sigma(t, n_steps))
    return (np.float32(1.0) - sg) * clean + sg * noise


def gen_do_head(wl: Workload, head: int, rows: int = 0) -> np.ndarray:
    """One head of the upstream gradient dO ~ N(0,1), float32 [rows or N, d] (block order;
    rows > N for a padded block order)."""
    return _rng(wl.cid, DO_ID, head).standard_normal((rows or wl.N, wl.d), dtype=np.float32)


def gen_a2v(wl: Workload) -> np.ndarray:
    """A2V feature-norm field over the raster token grid: float32 [N]."""
    rng = _rng(wl.cid, A2V_ID)
    T, H, W = wl.grid
    centres = rng.uniform(0.0, 1.0, size=(wl.bumps, 3)) * np.array([T, H, W], dtype=np.float64)
    t, h, w = _coords(wl.grid)
    field_ = np.zeros((T, H, W), dtype=np.float64)
    for c in centres:
        r2 = (t - c[0]) ** 2 + (h - c[1]) ** 2 + (w - c[2]) ** 2
        field_ += np.exp(-r2 / (2.0 * wl.sigma ** 2))
    return field_.reshape(-1).astype(np.float32)


def to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round to nearest even); returned as float32."""
    import torch

    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).float().numpy()


def round_inputs(wl: Workload, x: np.ndarray) -> np.ndarray:
    """The values the path actually sees: bf16-rounded for bf16 workloads, else float32."""
    return to_bf16(x) if wl.dtype == "bf16" else np.asarray(x, dtype=np.float32)


def gen_heads(wl: Workload, tensor: int, heads, threads: int = 8, rows: int = 0) -> list:
    """Several heads of one tensor, generated in parallel threads (numpy releases the GIL).
    rows: the block-order length of dO when it is not N (a padded block order)."""
    rope = rope_tables(wl.grid, wl.d, wl.rope_split) if tensor in (Q_ID, K_ID) else None

    def one(h):
        x = gen_do_head(wl, h, rows) if tensor == DO_ID else gen_head(wl, tensor, h, rope)
        return round_inputs(wl, x)

    with ThreadPoolExecutor(max_workers=threads) as ex:
        return list(ex.map(one, list(heads)))


def gen_scores(nb: int, rows: int, seed: int, scale: float = 1.0, ties: bool = False) -> np.ndarray:
    """Synthetic block-score rows float32 [rows, nb] for selection-only tests.

    Scores are normal with a per-row spread drawn from [0.05, 3] * scale, so that
    some rows are flat (the cumulative-mass cut dominates) and some peaked (the
    top-k count dominates).  With ``ties`` values are quantised to force exact ties.
    """
    rng = _rng(1000, seed)
    spread = rng.uniform(0.05, 3.0, size=(rows, 1)) * scale
    s = rng.standard_normal((rows, nb)) * spread
    if ties:
        s = np.round(s * 4.0) / 4.0
    return s.astype(np.float32)


def gen_block_lists(nb: int, heads: int, seed: int, min_keep: int = 1, max_keep: int = 0):
    """Seeded random kept-block lists (counts [heads, nb], idx [heads, nb, nb] ascending).

    Used to drive the attention kernels with lists independent of any selection code.
    """
    rng = _rng(2000, seed)
    max_keep = max_keep or nb
    counts = rng.integers(min_keep, max_keep + 1, size=(heads, nb)).astype(np.int32)
    idx = np.full((heads, nb, nb), -1, dtype=np.int32)
    for h in range(heads):
        for i in range(nb):
            sel = np.sort(rng.choice(nb, size=counts[h, i], replace=False))
            idx[h, i, : counts[h, i]] = sel
    return counts, idx
