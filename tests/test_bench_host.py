"""Host logic of bench.py that needs no GPU: the DRAM-traffic records it reads, the
workload labels, the whole-job throughput arithmetic and the oracle sample's work."""
import dataclasses
import json
import os

import bench
from audio_diffusion_dits_zone_b300 import synth


def test_dram_traffic_follows_the_source():
    # a capture counts only while its kernel's source file is the one captured
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        rows = json.load(f)["captures"]
    for r in rows:
        t, note = bench.dram_traffic(r["workload"], r["kernel"])
        if bench.source_sha1(r["source"]) == r["source_sha1"]:
            assert t == r["bytes_per_launch"] and t >= 0.99 * r["algorithmic_bytes"], r
        else:
            assert t is None and "changed" in note, r
    assert bench.dram_traffic("train720p", "no_such_kernel")[0] is None
    assert bench.dram_traffic("no_such_workload", "bsa_fwd_tc")[0] is None


def test_workload_labels_follow_the_mode():
    sp = 0.8
    assert "fwd+bwd" in bench.workload_config(synth.WORKLOADS["train720p"], sp)["workload"]
    c2k = bench.workload_config(synth.WORKLOADS["2k"], 0.93)["workload"]
    assert "forward only" in c2k and "head groups of 8" in c2k
    a = bench.a2v_config(synth.WORKLOADS["720p"], synth.AUDIO_TOKENS)
    assert a["audio_tokens"] == 157 and a["seq_len"] == 75600


def test_job_throughput_is_whole_job():
    # every rank processes its own replica: N ranks do N times the work in the same time
    assert bench.job_throughput(2e12, 1, 1.0) == 2.0
    assert bench.job_throughput(2e12, 4, 2.0) == 4.0


def test_oracle_sample_counts_the_work_of_the_mode():
    wl = synth.WORKLOADS["tiny"]
    ctx = bench.oracle_context(wl, 0)
    train = bench.oracle_sample_step(wl, wl.sparsity, ctx, [0, 5])
    fwd = bench.oracle_sample_step(dataclasses.replace(wl, mode="fwd"), wl.sparsity, ctx, [0, 5])
    assert train > 0 and abs(train / fwd - 14.0 / 4.0) < 1e-12


def test_oracle_sample_backward_is_the_full_backward_of_its_rows():
    # the sampled backward computes dK/dV contributions: on the tiny workload, sampling
    # every query block gives the full backward
    import numpy as np

    from oracle import prism_oracle as po

    wl = synth.WORKLOADS["tiny"]
    Qb, Kb, Vb, dO = bench.oracle_context(wl, 0)
    S = po.block_scores(po.block_mean(Qb, wl.block), po.block_mean(Kb, wl.block))
    counts, idx = po.select(S, wl.sparsity, wl.cdf_tau)
    O, L = po.bsa_forward(Qb, Kb, Vb, counts, idx, wl.block)
    full = po.bsa_backward(Qb, Kb, Vb, O, dO, L, counts, idx, wl.block)
    half1 = po.bsa_backward(Qb, Kb, Vb, O, dO, L, counts, idx, wl.block, qblocks=range(0, wl.nb, 2))
    half2 = po.bsa_backward(Qb, Kb, Vb, O, dO, L, counts, idx, wl.block, qblocks=range(1, wl.nb, 2))
    for f, a, b in zip(full, half1, half2):
        np.testing.assert_allclose(a + b, f, atol=1e-12)
        assert np.abs(a).sum() > 0
