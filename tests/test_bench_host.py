"""Host logic of bench.py that needs no GPU: the DRAM-traffic table it reads, the
workload labels, the whole-job throughput arithmetic and the oracle sample's work."""
import dataclasses

import bench
from audio_diffusion_dits_zone_b300 import synth


def test_dram_traffic_rows():
    t = bench.dram_traffic("train720p", "bsa_dkdv_tc")
    assert t is not None and t > 4.64e9  # at least the compulsory bytes
    assert bench.dram_traffic("a2v720p", "a2v_attn") > 7.7e8
    assert bench.dram_traffic("train720p", "no_such_kernel") is None
    assert bench.dram_traffic("no_such_workload", "bsa_dkdv_tc") is None


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
