"""The fused score + selection call against the two-call path (the scores of
prism_pool_score, then prism_select) on the same block means -- the lists must be equal
bit for bit, since the scores are summed in the same order and the selection rule and
its fixed-point masses are the same -- and against the oracle's selection (exact, or
within the stated tie rules)."""
import numpy as np
import pytest
import torch

from audio_diffusion_dits_zone_b300 import prism as P
from audio_diffusion_dits_zone_b300 import synth
from oracle import prism_oracle as po
from parity import check_lists, record, tie_budget

pytestmark = pytest.mark.gpu


def two_call(qb, kb, sp, tau):
    """Lists and fp32 scores from prism_pool_score (block size 1: the means are the rows
    themselves) and prism_select."""
    Hh, nb, d = qb.shape
    q = qb.permute(1, 0, 2).contiguous()  # [nb tokens, Hh, d]
    k = kb.permute(1, 0, 2).contiguous()
    qbar, kbar = torch.empty_like(qb), torch.empty_like(kb)
    S = torch.empty(Hh, nb, nb, device="cuda")
    P.prism_pool_score(q, k, None, None, 1, qbar=qbar, kbar=kbar, scores=S)
    counts = torch.empty(Hh, nb, dtype=torch.int32, device="cuda")
    idx = torch.full((Hh, nb, nb), -3, dtype=torch.int32, device="cuda")
    P.prism_select(S, sp, tau, counts, idx)
    assert torch.equal(qbar, qb) and torch.equal(kbar, kb)
    return counts, idx, S


def fused(qb, kb, sp, tau):
    Hh, nb, _ = qb.shape
    counts = torch.empty(Hh, nb, dtype=torch.int32, device="cuda")
    idx = torch.full((Hh, nb, nb), -3, dtype=torch.int32, device="cuda")
    P.prism_score_select(qb, kb, sp, tau, counts, idx)
    return counts, idx


def same_lists(c1, i1, c2, i2):
    assert torch.equal(c1, c2)
    c = c1.cpu().numpy()
    a, b = i1.cpu().numpy(), i2.cpu().numpy()
    for h in range(c.shape[0]):
        for i in range(c.shape[1]):
            n = c[h, i]
            assert np.array_equal(a[h, i, :n], b[h, i, :n]), (h, i)
            assert np.all(a[h, i, n:] == -3)  # untouched tail


def run_case(qb_np, kb_np, sp, tau, name):
    qb, kb = (torch.from_numpy(np.ascontiguousarray(x, np.float32)).cuda() for x in (qb_np, kb_np))
    c1, i1 = fused(qb, kb, sp, tau)
    c2, i2, S = two_call(qb, kb, sp, tau)
    assert P.status_check() == 0
    same_lists(c1, i1, c2, i2)
    S_ref = po.block_scores(qb_np.astype(np.float64), kb_np.astype(np.float64))
    err = np.abs(S.cpu().numpy() - S_ref).max(-1)
    stats, _ = check_lists(c1.cpu().numpy(), i1.cpu().numpy(), S_ref, sp, tau, score_err=err)
    record(f"score_select {name}", stats)
    return stats


@pytest.mark.parametrize("nb,Hh,d,sp", [(10, 2, 64, 0.75), (591, 2, 128, 0.8), (1339, 1, 128, 0.85),
                                        (2363, 1, 128, 0.93), (200, 3, 64, 0.0), (4096, 1, 64, 0.9), (37, 4, 8, 0.5)])
def test_score_select_matches_two_call_path_and_oracle(nb, Hh, d, sp):
    rng = np.random.default_rng(nb + d)
    spread = rng.uniform(0.05, 2.0, size=(Hh, nb, 1))
    qb = rng.normal(size=(Hh, nb, d)) * spread
    kb = rng.normal(size=(Hh, nb, d))
    stats = run_case(qb, kb, sp, 0.2, f"nb={nb} d={d} s={sp}")
    assert stats["score"] + stats["mass"] <= tie_budget(stats["rows"]), stats


def test_score_select_ties_flat_rows_and_refinement():
    nb, d = 1200, 64
    rng = np.random.default_rng(7)
    heads = []
    # head 0: keys from 5 distinct vectors (heavy exact ties); head 1: identical keys
    # (every row flat); head 2: a cluster of 900 keys within 1e-4 of one another plus
    # far outliers, so the crossing bucket holds far more than 256 blocks and is refined
    base = rng.normal(size=(5, d))
    heads.append(base[rng.integers(0, 5, nb)])
    heads.append(np.tile(rng.normal(size=(1, d)), (nb, 1)))
    u = rng.normal(size=d)
    k2 = u[None, :] + 1e-6 * rng.normal(size=(nb, d))
    k2[:300] = -5 * u[None, :] + rng.normal(size=(300, d))  # far below the cluster for queries along u
    heads.append(k2)
    kb = np.stack(heads)
    qb = rng.normal(size=(3, nb, d))
    qb[2] = np.abs(rng.normal(size=(nb, 1))) * u[None, :] + 0.01 * rng.normal(size=(nb, d))
    qb[1, :10] = 0.0  # rows of all-zero scores
    run_case(qb, kb, 0.93, 0.2, "ties/flat/refinement")
