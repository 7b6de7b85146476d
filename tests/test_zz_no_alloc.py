"""The workspace-free zone-shape entry point gives the same answer as the usual one.

prism_zone_shapes_noalloc exists for callers that cannot hand the library device
memory (their memory belongs to another allocator, or they run inside a hook that
must not allocate).  Its scratch is a fixed array inside the library, shared by all
calls, so this test runs it twice in a row on different grids and checks each
result against prism_zone_shapes with a caller workspace.  The outputs are integer
shape ids and a permutation, so they must agree exactly.  This file is collected
last so that a failure here never hides a failure elsewhere.
"""
import ctypes

import numpy as np
import pytest
import torch

from audio_diffusion_dits_zone_b300 import prism as P
from audio_diffusion_dits_zone_b300 import synth

pytestmark = pytest.mark.gpu


def _case(grid, zext, heads, d, dtype, cid):
    shapes = synth.SHAPES_128 if d == 128 else synth.SHAPES_64
    split = (44, 42, 42) if d == 128 else (16, 24, 24)
    wl = synth.Workload("noalloc", cid, grid, heads, d, dtype, zext, 128, shapes, 0.8, 0.2, 2, 3.0, split, "fwd")
    V = np.concatenate(synth.gen_heads(wl, synth.V_ID, range(heads)), axis=1)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    feat = torch.from_numpy(V).cuda().to(tdt)
    a2v = torch.from_numpy(synth.gen_a2v(wl)).cuda()
    Z = -(-grid[0] // zext[0]) * -(-grid[1] // zext[1]) * -(-grid[2] // zext[2])
    return wl, feat, a2v, Z


def test_noalloc_zone_shapes_match_workspace_version_twice():
    cases = [((7, 20, 40), (3, 9, 16), 3, 128, "bf16", 61), ((5, 8, 16), (5, 4, 8), 2, 64, "f32", 62)]
    for grid, zext, heads, d, dtype, cid in cases:
        wl, feat, a2v, Z = _case(grid, zext, heads, d, dtype, cid)
        zs_ref = torch.empty(Z, dtype=torch.int32, device="cuda")
        perm_ref = torch.empty(wl.N, dtype=torch.int32, device="cuda")
        P.prism_zone_shapes(feat, heads * d, a2v, grid, zext, wl.shapes, zs_ref, perm_ref)
        zs = torch.full((Z,), -1, dtype=torch.int32, device="cuda")
        perm = torch.full((wl.N,), -1, dtype=torch.int32, device="cuda")
        P.prism_zone_shapes_noalloc(feat, heads * d, a2v, grid, zext, wl.shapes, zs, perm)
        assert P.status_check() == 0
        assert torch.equal(zs, zs_ref), grid
        assert torch.equal(perm, perm_ref), grid


def test_noalloc_rejects_grids_beyond_its_scratch():
    # 700 zones x 40,000 channels would need about 5 MB of scratch: refused before any
    # device work.  The device pointers are NULL, so a regression of the size check
    # ends in the NULL-pointer refusal (PRISM_EINVAL), never in a launch.
    shapes = (ctypes.c_int32 * 12)(1, 8, 16, 2, 8, 8, 4, 4, 8, 8, 4, 4)
    rc = P.lib().prism_zone_shapes_noalloc(None, P.PRISM_BF16, 40000, 40000, None, 21, 90, 160, 3, 9, 16, shapes,
                                           4, None, None, None)
    assert rc == P.PRISM_EUNSUPPORTED
    assert b"scratch" in P.lib().prism_last_error()
