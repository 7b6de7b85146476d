"""GPU parity of prism_a2v_norm (audio-to-video cross-attention and its per-token
feature norm) against the CPU oracle, on seeded inputs: small grids element by
element, with ragged audio and video tails, and the full 720p grid on sampled rows."""
import numpy as np
import pytest
import torch

from audio_diffusion_dits_zone_b300 import prism as P
from audio_diffusion_dits_zone_b300 import synth
from oracle import prism_oracle as po
from parity import attn_close

pytestmark = pytest.mark.gpu
dev = "cuda"


def workload(grid, heads, cid):
    return synth.Workload("a2v", cid, grid, heads, 128, "bf16", (3, 9, 16), 128, synth.SHAPES_128, 0.8, 0.2, 1, 3.0,
                          (44, 42, 42), "fwd")


def to_dev(x):
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(dev).to(torch.bfloat16)


def check_field(got, ref, what):
    # a2v is a norm of an attention output whose entries meet the attention tolerances
    # (max-abs 2e-2, mean-abs 2e-3); relative to the norm that is well inside 1e-2
    rel = np.abs(got - ref) / np.maximum(ref, 1e-6)
    assert rel.max() < 1e-2, (what, rel.max(), int(rel.argmax()))
    assert rel.mean() < 1e-3, (what, rel.mean())


@pytest.mark.parametrize("grid,heads,M", [((5, 8, 16), 2, 157),   # 640 video tokens, audio 128 + 29
                                          ((3, 9, 17), 3, 128),   # 459 video tokens (ragged), one audio block
                                          ((2, 5, 13), 1, 1),     # one audio token: O = Va[0] everywhere
                                          ((3, 8, 16), 2, 40),    # two 32-key chunks, the second short
                                          ((3, 8, 16), 2, 70),    # three chunks
                                          ((5, 16, 32), 16, 157),  # 320 tiles: CTAs walk several, across heads
                                          ((4, 8, 16), 2, 300)])  # three audio blocks (the general kernel)
def test_a2v_matches_oracle(grid, heads, M):
    wl = workload(grid, heads, 60 + M % 7)
    qv, ka, va = synth.gen_a2v_inputs(wl, range(heads), M)
    N = wl.N
    a2v = torch.empty(N, device=dev)
    o = torch.empty(N, heads, 128, device=dev, dtype=torch.bfloat16)
    P.prism_a2v_norm(to_dev(qv), to_dev(ka), to_dev(va), a2v, o)
    assert P.status_check() == 0
    ref, O = po.a2v_field(qv, ka, va)
    attn_close(o.float().cpu().numpy(), O, what="a2v O")
    check_field(a2v.cpu().numpy(), ref, "a2v")


def test_a2v_without_output_and_strided_views():
    # o = NULL (only the field), and q / k / v as head-sliced views of wider rows
    wl = workload((3, 9, 16), 4, 70)
    qv, ka, va = synth.gen_a2v_inputs(wl, range(4), 157)
    wide_q = torch.zeros(wl.N, 6, 128, device=dev, dtype=torch.bfloat16)
    wide_k = torch.zeros(157, 6, 128, device=dev, dtype=torch.bfloat16)
    wide_v = torch.zeros(157, 6, 128, device=dev, dtype=torch.bfloat16)
    wide_q[:, 1:5] = to_dev(qv)
    wide_k[:, 2:6] = to_dev(ka)
    wide_v[:, 2:6] = to_dev(va)
    a2v = torch.empty(wl.N, device=dev)
    P.prism_a2v_norm(wide_q[:, 1:5], wide_k[:, 2:6], wide_v[:, 2:6], a2v)
    assert P.status_check() == 0
    check_field(a2v.cpu().numpy(), po.a2v_field(qv, ka, va)[0], "a2v strided")


def test_a2v_rejects_unsupported():
    q = torch.zeros(64, 1, 64, device=dev, dtype=torch.bfloat16)
    a2v = torch.empty(64, device=dev)
    with pytest.raises(P.PrismError) as e:
        P.prism_a2v_norm(q, q[:8], q[:8], a2v)
    assert e.value.code == 2  # PRISM_EUNSUPPORTED: d = 64


def test_a2v_full_720p_sampled_rows():
    # the 720p grid, 40 heads, 157 audio tokens: the launch the bench times, checked on
    # 512 rows spread over the sequence (the oracle computes them one by one)
    wl = synth.WORKLOADS["720p"]
    qv, ka, va = synth.gen_a2v_inputs(wl, range(wl.heads))
    a2v = torch.empty(wl.N, device=dev)
    P.prism_a2v_norm(to_dev(qv), to_dev(ka), to_dev(va), a2v)
    assert P.status_check() == 0
    rows = np.linspace(0, wl.N - 1, 512).astype(np.int64)
    ref, _ = po.a2v_field(qv, ka, va, rows=rows)
    check_field(a2v.cpu().numpy()[rows], ref, "a2v 720p")
