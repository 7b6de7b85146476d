"""Benchmark of one Prism block-sparse attention layer, forward + backward, on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload train720p] [--sparsity 0.8]

A step is one pass of the whole path over one batch of synthetic input: zone
shapes -> pool + score -> hybrid select -> block-sparse attention forward ->
backward, for all heads of one layer.  Default workload: the 720p training step
(T=21, H=45, W=80 = 75,600 tokens, 40 heads, d = 128, bf16, sparsity 0.80, CDF 0.20).
Inputs are generated from seeds, copied to HBM before timing, and are larger than
L2 (Q, K, V, dO: 774 MB each), so no flush is needed between steps.

Prints one JSON line (rank 0).  value = executed-block attention TFLOP/s of the
whole step (forward 4*|b_i|*|b_j|*d + backward 10*|b_i|*|b_j|*d per kept block
pair, divided by the step time); for N GPUs (torchrun) every rank runs its own
replica of the workload and value = total work / max-over-ranks time.
--impl reference times the CPU oracle on the host cores on a bounded sample.

--workload a2v720p times the step upstream of the path instead: the audio-to-video
cross-attention of the 720p grid's 75,600 video tokens over 157 audio tokens (40
heads, d = 128, bf16) and its per-token feature norm, the A2V field the zone step
reads; value = its TFLOP/s (4 * N * M * d * heads per call).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "block-sparse attn fwd+bwd ms/layer & effective TFLOPS (% bf16 peak), 720p–2K"
UNIT = "TFLOP/s"


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16": d["bf16_tflops"], "bf16_sustained": d["bf16_tflops_sustained"],
                "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16": 1800.0, "bf16_sustained": 1400.0, "source": "fallback"}


def workload_config(wl, sparsity):
    what = "fwd+bwd" if wl.mode == "fwd+bwd" else "forward only (as the config specifies)"
    groups = f", attention in head groups of {wl.head_group}" if wl.head_group else ""
    return {"workload": f"{wl.name}: Prism layer {what}{groups}, T={wl.grid[0]},H={wl.grid[1]},W={wl.grid[2]} "
                        f"({wl.N} tokens), {wl.heads} heads, d={wl.d}, {wl.dtype}, B={wl.block}, "
                        f"zones {wl.zone[0]}x{wl.zone[1]}x{wl.zone[2]}, sparsity {sparsity}, CDF {wl.cdf_tau}",
            "global_batch": 1, "seq_len": wl.N, "heads": wl.heads, "head_dim": wl.d, "sparsity": sparsity,
            "cdf_tau": wl.cdf_tau, "parallelism": "replicas (one layer per GPU)",
            "l2": "inputs larger than L2 (Q, K, V, dO 774 MB each); no flush"}


# ------------------------------------------------------------ multi-rank
def max_over_ranks(x: float, device) -> float:
    """The largest value of x over all ranks (the job's time is its slowest rank's)."""
    import torch

    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(work_per_rank: float, world: int, seconds: float) -> float:
    """Whole-job TFLOP/s: every rank processes its own replica of the workload."""
    return world * work_per_rank / seconds / 1e12


def source_sha1(rel):
    """SHA-1 of a source file of the repository (to tie a capture to the code it measured)."""
    import hashlib

    path = os.path.join(ROOT, rel)
    if not os.path.exists(path):
        return None
    with open(path, "rb") as f:
        return hashlib.sha1(f.read()).hexdigest()


def dram_traffic(workload, kernel):
    """(bytes, note): DRAM bytes (read + write) per launch of `kernel` on `workload` from
    the ncu capture recorded in profiles/traffic.json, and where that figure comes from.
    bytes is None when no capture is recorded, or when the kernel's source file has
    changed since the capture (its SHA-1 differs from the one recorded with it)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None, "no ncu capture recorded"
    with open(path) as f:
        rows = json.load(f)["captures"]
    for r in rows:
        if r["workload"] == workload and r["kernel"] == kernel:
            if source_sha1(r["source"]) != r["source_sha1"]:
                return None, f"{r['source']} changed since the ncu capture"
            return float(r["bytes_per_launch"]), f"ncu capture: {r['capture']}"
    return None, "no ncu capture of this kernel as it stands"


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [x.strip() for x in line.split(",")]
                    if len(parts) >= 9:
                        rows.append(parts)
        finally:
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = max(float(r[2]) for r in rows if r[2].replace(".", "").isdigit())
        load = [s for s in sm if s > 0.5 * mx] or sm
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(load), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(rows), "power_w_max": max(float(r[3]) for r in rows if r[3].replace(".", "").isdigit())}


# ----------------------------------------------------------------- ours
def run_ours(args, rank, world, local_rank):
    import numpy as np
    import torch

    from audio_diffusion_dits_zone_b300 import prism as P
    from audio_diffusion_dits_zone_b300 import synth
    from audio_diffusion_dits_zone_b300.pipeline import PrismLayer

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    wl = synth.WORKLOADS[args.workload]
    sp = wl.sparsity if args.sparsity is None else args.sparsity
    train = wl.mode == "fwd+bwd"
    layer = PrismLayer(wl, dev, sparsity=sp, train=train, fused_select=args.select == "fused",
                       chunked=args.blocks == "zone-chunked")
    layer.load_inputs()
    layer.step()
    if P.status_check() != 0:
        raise RuntimeError("device status word set after the first step")
    fwd_fl, bwd_fl, dense_f, dense_b = layer.flops()
    if not train:  # forward-only configurations: the step ends with the forward
        bwd_fl = dense_b = 0.0
    work = fwd_fl + bwd_fl
    names = ["zone_shapes", "pool_score", "select", "bsa_fwd"] + (["bsa_bwd"] if train else [])
    calls = [layer.zone_shapes, layer.pool_score, layer.select, layer.attention_fwd] + \
        ([layer.attention_bwd] if train else [])
    for _ in range(args.warmup):
        layer.step()
    torch.cuda.synchronize()
    # ---------------- timed region: K steps; events around every call and every kernel,
    # all recorded on the launching stream (torch's current stream)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)] for _ in range(args.steps)]
    launches0 = P.launch_count()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk, P.KernelTimer() as kt:
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record()
        for s in range(args.steps):
            ev[s][0].record()
            for c, fn in enumerate(calls):
                fn()
                ev[s][c + 1].record()
        t1.record()
        torch.cuda.synchronize()
    launches = P.launch_count() - launches0
    elapsed_ms = t0.elapsed_time(t1)
    if world > 1:
        elapsed_ms = max_over_ranks(elapsed_ms, dev)
        torch.distributed.barrier()
    if P.status_check() != 0:
        raise RuntimeError("device status word set during the timed region")
    per_call = {n: statistics.mean(ev[s][c].elapsed_time(ev[s][c + 1]) for s in range(args.steps))
                for c, n in enumerate(names)}
    kdur = kt.durations()
    per_kernel = {n: {"ms_per_step": round(sum(v) / args.steps, 4), "launches_per_step": len(v) // args.steps,
                      "ms_per_launch": round(statistics.mean(v), 4)} for n, v in kdur.items()}
    ms = elapsed_ms / args.steps
    pk = peaks()
    value = job_throughput(work, world, ms * 1e-3)

    # algorithmic work of each kernel per step: the matmul FLOPs it performs
    # (tensor-bound kernels) or the bytes it must move (memory-bound kernels)
    pairs = fwd_fl / (4.0 * wl.d)
    C = wl.heads * wl.d
    kept = int(layer.counts.sum().item())
    nb, R = layer.nb, layer.nrows
    algo = {
        "bsa_fwd_tc": ("tensor", 4.0 * pairs * wl.d), "bsa_dq_tc": ("tensor", 6.0 * pairs * wl.d),
        "bsa_dkdv_tc": ("tensor", 8.0 * pairs * wl.d), "bsa_bwd_tc": ("tensor", 10.0 * pairs * wl.d),
        "dq_convert": ("hbm", wl.heads * R * wl.d * 4.0 + R * C * 2.0),
        "zone_tma": ("hbm", wl.N * C * 2.0), "zone_partial": ("hbm", wl.N * C * 2.0),
        "pool_gather": ("hbm", 3.0 * wl.N * C * 2 + 3.0 * R * C * 2 + 2.0 * wl.heads * nb * wl.d * 4),
        "scores": ("hbm", wl.heads * nb ** 2 * 4.0 + 2.0 * wl.heads * nb * wl.d * 4),
        "score_select": ("hbm", 2.0 * wl.heads * nb * wl.d * 4 + wl.heads * nb * 4 + 4.0 * kept),
        "select": ("hbm", wl.heads * nb ** 2 * 4.0 + wl.heads * nb * 4 + 4.0 * kept),
        "bwd_prep": ("hbm", 2.0 * R * C * 2 + wl.heads * R * 4 + 2.0 * wl.heads * nb * wl.block * 4),
    }
    for n, (bound, w) in algo.items():
        if n in per_kernel:
            t = per_kernel[n]["ms_per_step"] * 1e-3
            if bound == "tensor":
                per_kernel[n]["TFLOP/s"] = round(w / t / 1e12, 2)
                per_kernel[n]["frac_bf16_burst"] = round(w / t / 1e12 / pk["bf16"], 4)
                per_kernel[n]["frac_bf16_sustained"] = round(w / t / 1e12 / pk["bf16_sustained"], 4)
            else:
                per_kernel[n]["GB/s"] = round(w / t / 1e9, 1)
                per_kernel[n]["frac_hbm"] = round(w / t / 1e9 / pk["hbm_gbs"], 4)
    # the score GEMM on CUDA cores against the fp32 FMA peak: SMs x 128 lanes x 2 FLOP x clock
    # (the maximum SM clock, and the median one sampled under load)
    clocks = clk.summary()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    score_flops = 2.0 * wl.heads * nb ** 2 * wl.d
    for n in ("scores", "score_select"):
        if n in per_kernel:
            t = per_kernel[n]["ms_per_step"] * 1e-3
            achieved = score_flops / t / 1e12
            per_kernel[n]["fp32_TFLOP/s"] = round(achieved, 2)
            if clocks.get("sm_max_mhz"):
                peak_max = sms * 128 * 2 * clocks["sm_max_mhz"] * 1e6 / 1e12
                per_kernel[n]["frac_fp32_alu"] = round(achieved / peak_max, 4)
                per_kernel[n]["fp32_alu_peak"] = f"{peak_max:.1f} TFLOP/s at {clocks['sm_max_mhz']:.0f} MHz"
            if clocks.get("sm_mhz"):
                per_kernel[n]["frac_fp32_alu_at_median_clock"] = round(
                    achieved / (sms * 128 * 2 * clocks["sm_mhz"] * 1e6 / 1e12), 4)
    dom = max(per_kernel, key=lambda n: per_kernel[n]["ms_per_step"])
    bound, w = algo.get(dom, ("tensor", 0.0))
    t_launch = per_kernel[dom]["ms_per_launch"] * 1e-3
    w_launch = w / max(1, per_kernel[dom]["launches_per_step"])
    traffic, traffic_note = dram_traffic(wl.name, dom)
    if bound == "tensor":
        # the burst peak: kernels of this step run above the seconds-long sustained figure
        achieved = w_launch / t_launch / 1e12
        roofline = {"bound": "tensor", "kernel": dom, "achieved": round(achieved, 2), "peak": pk["bf16"],
                    "unit": "TFLOP/s", "frac": round(achieved / pk["bf16"], 4), "traffic": traffic,
                    "traffic_note": traffic_note,
                    "peak_note": f"bf16 dense, burst ({pk['source']}); sustained {pk['bf16_sustained']}",
                    "frac_of_sustained": round(achieved / pk["bf16_sustained"], 4),
                    "algorithmic_per_launch": f"{w_launch:.4e} FLOP"}
    else:
        achieved = w_launch / t_launch / 1e9
        roofline = {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": pk["hbm_gbs"],
                    "unit": "GB/s", "frac": round(achieved / pk["hbm_gbs"], 4), "traffic": traffic,
                    "traffic_note": traffic_note}

    # ---------------- end to end through the public API, host buffers
    e2e = None if args.no_e2e else run_e2e(layer, args, world)
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded Wan-VAE-shaped latents, no weights)",
        "config": {**workload_config(wl, sp), "blocks": args.blocks, "select": args.select,
                   "backward": "fused" if os.environ.get("PRISM_BWD_FUSED") == "1" else "split"},
        "ms_per_layer": round(ms, 3),
        "tflops_executed": round(work / (ms * 1e-3) / 1e12, 3),
        "tflops_dense_equivalent": round((dense_f + dense_b) / (ms * 1e-3) / 1e12, 3),
        "pct_bf16_peak_executed": round(100 * work / (ms * 1e-3) / 1e12 / pk["bf16"], 2),
        "pct_bf16_sustained_executed": round(100 * work / (ms * 1e-3) / 1e12 / pk["bf16_sustained"], 2),
        "per_call_ms": {n: round(v, 4) for n, v in per_call.items()},
        "per_kernel": per_kernel,
        "attention_tflops": {"bsa_fwd": round(fwd_fl / (per_call["bsa_fwd"] * 1e-3) / 1e12, 2),
                             **({"bsa_bwd": round(bwd_fl / (per_call["bsa_bwd"] * 1e-3) / 1e12, 2)} if train else {})},
        "kept_fraction": round(float(layer.counts.double().mean().item()) / layer.nb, 4),
        "roofline": roofline,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clocks,
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(wl, sp, budget_s=args.cpu_seconds)
    return line


def run_e2e(layer, args, world):
    """Same step through the public API with host buffers.  Every step copies its
    inputs (Q, K, V, A2V field, and dO when training) from pinned host memory to the
    device and its results (O, and dQ, dK, dV when training) back to pinned host memory.  Two device layers take the
    steps in turn so that the copies of one step overlap the compute of the other:
    host-to-device copies on one stream, the library calls on a second, device-to-host
    copies on a third, ordered by events (a layer's inputs are refilled only after
    the step that read them, its outputs rewritten only after they were copied out).
    Within a step the forward waits only for its own inputs (dO follows) and O is
    copied out while the backward runs."""
    import torch

    from audio_diffusion_dits_zone_b300.pipeline import PrismLayer

    layers = [layer, PrismLayer(layer.wl, layer.device, sparsity=layer.sparsity, train=layer.train,
                                fused_select=layer.fused_select, chunked=layer.chunked)]

    def ins(L):
        return [L.q, L.k, L.v, L.a2v] + ([L.do_blk] if L.train else [])

    def outs(L):
        return [L.o_blk] + ([L.dq, L.dk, L.dv] if L.train else [])

    n_fwd_in = 4  # Q, K, V and the A2V field feed the forward; dO only the backward
    h_in = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in ins(layer)]
    for h, t in zip(h_in, ins(layer)):
        h.copy_(t)
    h_out = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs(layer)] for _ in range(2)]
    s_in, s_run, s_out = (torch.cuda.Stream(layer.device) for _ in range(3))
    # the first step's inputs and the last step's outputs cannot overlap compute: time
    # enough steps (about two seconds of work) for the steady state to dominate
    steps = max(20, min(args.steps, 40))

    def run(n):
        ran, out = [None, None], [None, None]
        for s in range(n):
            L, x = layers[s & 1], s & 1
            e_fwd, e_bwd, f_done = torch.cuda.Event(), torch.cuda.Event(), torch.cuda.Event()
            with torch.cuda.stream(s_in):
                if ran[x] is not None:
                    s_in.wait_event(ran[x])
                for i, (h, t) in enumerate(zip(h_in, ins(L))):
                    t.copy_(h, non_blocking=True)
                    if i == n_fwd_in - 1:
                        e_fwd.record(s_in)
                e_bwd.record(s_in)
            with torch.cuda.stream(s_run):
                s_run.wait_event(e_fwd)
                if out[x] is not None:
                    s_run.wait_event(out[x])
                L.forward(s_run)
                f_done.record(s_run)
                if L.train:
                    s_run.wait_event(e_bwd)
                    L.attention_bwd(s_run)
                ran[x] = torch.cuda.Event()
                ran[x].record(s_run)
            with torch.cuda.stream(s_out):
                # O is final after the forward: it leaves while the backward runs
                s_out.wait_event(f_done)
                h_out[x][0].copy_(outs(L)[0], non_blocking=True)
                s_out.wait_event(ran[x])
                for h, t in zip(h_out[x][1:], outs(L)[1:]):
                    h.copy_(t, non_blocking=True)
                out[x] = torch.cuda.Event()
                out[x].record(s_out)
        torch.cuda.synchronize(layer.device)

    run(2)
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    run(steps)
    dt = (time.perf_counter() - t0) / steps
    if world > 1:
        dt = max_over_ranks(dt, layer.device)
    fwd_fl, bwd_fl, _, _ = layer.flops()
    if not layer.train:
        bwd_fl = 0.0
    del layers[1]
    return {"value": round(world * (fwd_fl + bwd_fl) / dt / 1e12, 3), "unit": UNIT, "ms_per_step": round(dt * 1e3, 3),
            "h2d_bytes_per_step": int(sum(t.numel() * t.element_size() for t in ins(layer))),
            "d2h_bytes_per_step": int(sum(t.numel() * t.element_size() for t in outs(layer))), "steps": steps,
            "overlap": "two device layers alternate; H2D, compute and D2H on three streams; the forward starts "
                       "once Q, K, V and the A2V field have landed and O leaves while the backward runs"}


# ------------------------------------------------------------ A2V field
A2V_METRIC = "A2V cross-attention + feature norm ms/call & TFLOPS (% bf16 peak), 720p"


def a2v_config(wl, M):
    return {"workload": f"a2v720p: audio-to-video cross-attention + per-token feature norm, video grid "
                        f"T={wl.grid[0]},H={wl.grid[1]},W={wl.grid[2]} ({wl.N} tokens), {M} audio tokens, "
                        f"{wl.heads} heads, d={wl.d}, bf16",
            "global_batch": 1, "seq_len": wl.N, "audio_tokens": M, "heads": wl.heads, "head_dim": wl.d,
            "parallelism": "replicas (one layer per GPU)",
            "l2": "video queries larger than L2 (774 MB); no flush"}


def run_a2v(args, rank, world, local_rank):
    import torch

    from audio_diffusion_dits_zone_b300 import prism as P
    from audio_diffusion_dits_zone_b300 import synth

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    wl, M = synth.WORKLOADS["720p"], synth.AUDIO_TOKENS
    qv_h, ka_h, va_h = synth.gen_a2v_inputs(wl, range(wl.heads), M)
    qv, ka, va = (torch.from_numpy(x).to(dev).to(torch.bfloat16) for x in (qv_h, ka_h, va_h))
    a2v = torch.empty(wl.N, device=dev)
    ws = P.prism_a2v_norm(qv, ka, va, a2v)
    for _ in range(args.warmup):
        P.prism_a2v_norm(qv, ka, va, a2v, ws=ws)
    if P.status_check() != 0:
        raise RuntimeError("device status word set in the warm-up")
    steps = max(args.steps, 20)  # ~0.3 ms per call: enough calls for a stable mean
    launches0 = P.launch_count()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clk, P.KernelTimer() as kt:
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record()
        for _ in range(steps):
            P.prism_a2v_norm(qv, ka, va, a2v, ws=ws)
        t1.record()
        torch.cuda.synchronize()
    launches = P.launch_count() - launches0
    ms = t0.elapsed_time(t1) / steps
    if world > 1:
        ms = max_over_ranks(ms, dev)
    if P.status_check() != 0:
        raise RuntimeError("device status word set during the timed region")
    flops = 4.0 * wl.N * M * wl.d * wl.heads              # algorithmic: the audio tokens that exist
    executed = 4.0 * wl.N * (-(-M // 128) * 128) * wl.d * wl.heads  # the key blocks the tensor cores run
    pk = peaks()
    kd = kt.durations()
    per_kernel = {n: {"ms_per_step": round(sum(v) / steps, 4), "launches_per_step": len(v) // steps,
                      "ms_per_launch": round(statistics.mean(v), 4)} for n, v in kd.items()}
    t_attn = per_kernel["a2v_attn"]["ms_per_launch"] * 1e-3
    achieved = flops / t_attn / 1e12
    per_kernel["a2v_attn"]["TFLOP/s"] = round(achieved, 2)
    per_kernel["a2v_attn"]["TFLOP/s_executed_blocks"] = round(executed / t_attn / 1e12, 2)
    bytes_attn = wl.N * wl.heads * wl.d * 2 + 2 * M * wl.heads * wl.d * 2 + wl.heads * wl.N * 4
    per_kernel["a2v_attn"]["GB/s"] = round(bytes_attn / t_attn / 1e9, 1)
    t_red = per_kernel["a2v_reduce"]["ms_per_launch"] * 1e-3
    per_kernel["a2v_reduce"]["GB/s"] = round((wl.heads * wl.N * 4 + wl.N * 4) / t_red / 1e9, 1)
    traffic, traffic_note = dram_traffic("a2v720p", "a2v_attn")
    roofline = {"bound": "tensor", "kernel": "a2v_attn", "achieved": round(achieved, 2), "peak": pk["bf16"],
                "unit": "TFLOP/s", "frac": round(achieved / pk["bf16"], 4), "traffic": traffic,
                "traffic_note": traffic_note,
                "peak_note": f"bf16 dense, burst ({pk['source']}; a 0.3 ms kernel between idle gaps); "
                             f"sustained {pk['bf16_sustained']}",
                "algorithmic_per_launch": f"{flops:.4e} FLOP ({M} audio tokens; the kernel runs "
                                          f"{-(-M // 128)} key blocks of 128)"}
    # end to end through the public call: video queries and audio keys / values copied in
    # from pinned host memory, the field copied back, every call
    hq, hk, hv = (torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (qv, ka, va))
    hq.copy_(qv), hk.copy_(ka), hv.copy_(va)
    ha = torch.empty(wl.N, dtype=torch.float32, pin_memory=True)
    e_steps = 5
    torch.cuda.synchronize()
    tt = time.perf_counter()
    for _ in range(e_steps):
        qv.copy_(hq, non_blocking=True)
        ka.copy_(hk, non_blocking=True)
        va.copy_(hv, non_blocking=True)
        P.prism_a2v_norm(qv, ka, va, a2v, ws=ws)
        ha.copy_(a2v, non_blocking=True)
    torch.cuda.synchronize()
    e_dt = (time.perf_counter() - tt) / e_steps
    if world > 1:
        e_dt = max_over_ranks(e_dt, dev)
    line = {"metric": A2V_METRIC, "value": round(world * flops / (ms * 1e-3) / 1e12, 3), "unit": UNIT,
            "n_gpus": world, "steps": steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded video queries, audio keys and values; no weights)",
            "config": a2v_config(wl, M), "per_kernel": per_kernel, "roofline": roofline,
            "e2e": {"value": round(world * flops / e_dt / 1e12, 3), "unit": UNIT, "ms_per_step": round(e_dt * 1e3, 3),
                    "h2d_bytes_per_step": int(sum(t.numel() * t.element_size() for t in (qv, ka, va))),
                    "d2h_bytes_per_step": int(a2v.numel() * 4), "steps": e_steps},
            "gpu_launches": launches, "clocks": clk.summary()}
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = a2v_cpu_baseline(qv_h, ka_h, va_h, budget_s=min(args.cpu_seconds, 10.0))
    return line


def a2v_cpu_baseline(qv, ka, va, budget_s=10.0):
    """The oracle's A2V field, timed on the host cores on rows spread over the grid:
    chunks of 256 evenly spaced rows, each chunk offset by one row from the last."""
    import numpy as np

    from oracle import prism_oracle as po

    N, Hh, d = qv.shape
    M = ka.shape[0]
    chunk, done, t0 = 256, 0, time.perf_counter()
    base = np.linspace(0, max(0, N - 1 - chunk), chunk).astype(np.int64)  # + offset < chunk stays below N
    while time.perf_counter() - t0 < budget_s and done + chunk <= N:
        po.a2v_field(qv, ka, va, rows=np.minimum(base + (done // chunk) % chunk, N - 1))
        done += chunk
    dt = time.perf_counter() - t0
    return {"value": round(4.0 * done * M * d * Hh / dt / 1e12, 6), "unit": UNIT, "cores": cpu_threads(),
            "kind": "oracle", "sample": f"{done} video rows (of {N}) spread over the grid, all {Hh} heads, "
                                        f"{M} audio tokens; {dt:.1f} s of CPU time; fp64 numpy"}


def run_a2v_reference(args):
    """--impl reference for the A2V workload: the oracle on bounded row samples."""
    from audio_diffusion_dits_zone_b300 import synth

    wl, M = synth.WORKLOADS["720p"], synth.AUDIO_TOKENS
    qv, ka, va = synth.gen_a2v_inputs(wl, range(wl.heads), M)
    a2v_cpu_baseline(qv, ka, va, budget_s=0.5 * max(1, args.warmup))
    per = max(2.0, min(20.0, 60.0 / max(1, args.steps)))
    res = [a2v_cpu_baseline(qv, ka, va, budget_s=per) for _ in range(args.steps)]
    v = statistics.mean(r["value"] for r in res)
    return {"metric": A2V_METRIC, "value": round(v, 6), "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(4.0 * wl.N * M * wl.d * wl.heads / (v * 1e12) * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": a2v_config(wl, M), "impl": "reference",
            "cpu_baseline": {"value": round(v, 6), "unit": UNIT, "cores": res[0]["cores"], "kind": "oracle",
                             "sample": f"each step: {res[0]['sample']}"},
            "e2e": {"value": round(v, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ------------------------------------------------- attention broadcast
PAB_METRIC = "Prism attention layer with attention broadcast across diffusion steps: ms per denoising step, 720p"
PAB_STEPS, PAB_RANGE = 30, 2


def run_pab(args, rank, world, local_rank):
    """A 30-step denoising trajectory of the 720p forward layer (zone shapes -> pool +
    score -> select -> forward on every computed step) with attention broadcast: the
    middle 70% of the steps compute attention every third step and reuse the output
    in between.  Timed twice, with the broadcast schedule and computing every step;
    value = ms per step with broadcast.  An untimed calibration pass measures the MSE
    between consecutive steps' outputs (selection held) with the library's kernel."""
    import numpy as np
    import torch

    from audio_diffusion_dits_zone_b300 import pab
    from audio_diffusion_dits_zone_b300 import prism as P
    from audio_diffusion_dits_zone_b300 import synth
    from audio_diffusion_dits_zone_b300.pipeline import PrismLayer

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    wl, n = synth.WORKLOADS["720p"], PAB_STEPS
    layer = PrismLayer(wl, dev, train=False)
    layer.load_inputs()
    # every step's Q, K, V resident before timing: (1 - sigma) x + sigma e, rounded to bf16
    steps = [[None] * 3 for _ in range(n)]
    for j, (tid, x) in enumerate(((synth.Q_ID, layer.q), (synth.K_ID, layer.k), (synth.V_ID, layer.v))):
        e = torch.empty(wl.N, wl.heads, wl.d, dtype=torch.float32, device=dev)
        for h0 in range(0, wl.heads, 8):
            hs = list(range(h0, min(h0 + 8, wl.heads)))
            for h, a in zip(hs, synth.gen_noise_heads(wl, tid, hs)):
                e[:, h].copy_(torch.from_numpy(a))
        xf = x.float()
        for t in range(n):
            sg = synth.trajectory_sigma(t, n)
            steps[t][j] = ((1.0 - sg) * xf + sg * e).to(torch.bfloat16)
        del e, xf
    torch.cuda.synchronize()

    def set_step(t):
        layer.q, layer.k, layer.v = steps[t]

    # calibration (untimed): consecutive-step MSE with the selection of step 0 held
    with P.KernelTimer() as kt_cal:
        curve = pab.calibrate(layer, set_step, n).double().mean(1).cpu().numpy()
    mse_ms = statistics.mean(kt_cal.durations()["attn_mse"])
    mse_bytes = 2.0 * wl.N * wl.heads * wl.d * 2

    def trajectory(rng):
        bl = pab.BroadcastLayer(layer, n, rng, "outputs")
        for t in range(n):
            set_step(t)
            bl.run_step(t)
        return sum(bl.plan)

    for _ in range(max(1, args.warmup // 3)):
        trajectory(PAB_RANGE)
    torch.cuda.synchronize()
    if P.status_check() != 0:
        raise RuntimeError("device status word set in the warm-up")
    res = {}
    launches0 = P.launch_count()
    with ClockSampler(local_rank) as clk:
        for rng in (PAB_RANGE, 0):
            if world > 1:
                torch.distributed.barrier()
            torch.cuda.synchronize()
            t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0.record()
            computed = trajectory(rng)
            t1.record()
            torch.cuda.synchronize()
            ms = t0.elapsed_time(t1)
            if world > 1:
                ms = max_over_ranks(ms, dev)
            res[rng] = (ms / n, computed)
    launches = P.launch_count() - launches0
    if P.status_check() != 0:
        raise RuntimeError("device status word set during the timed region")
    pk = peaks()
    ms_pab, comp = res[PAB_RANGE]
    ms_all = res[0][0]
    third = max(1, len(curve) // 3)
    line = {"metric": PAB_METRIC, "value": round(ms_pab, 3), "unit": "ms/step", "n_gpus": world, "steps": n,
            "warmup": args.warmup, "ms_per_step": round(ms_pab, 3), "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded Wan-VAE-shaped latents blended with seeded noise along a 30-step linear path)",
            "config": {"workload": f"pab720p: 720p Prism forward layer (T=21,H=45,W=80, {wl.N} tokens, {wl.heads} heads, "
                                   f"d={wl.d}, bf16, sparsity {wl.sparsity}, CDF {wl.cdf_tau}) over a {n}-step "
                                   f"denoising trajectory, attention broadcast range {PAB_RANGE} in the middle 70%",
                       "global_batch": 1, "seq_len": wl.N, "parallelism": "replicas (one layer per GPU)",
                       "l2": "inputs larger than L2 (every step's Q, K, V resident, 774 MB each); no flush"},
            "computed_steps": comp, "ms_per_step_every_step": round(ms_all, 3),
            "speedup_vs_every_step": round(ms_all / ms_pab, 3),
            "mse_consecutive_steps": {"first_third": float(curve[:third].mean()),
                                      "middle_third": float(curve[third:-third].mean()),
                                      "last_third": float(curve[-third:].mean())},
            "roofline": {"bound": "hbm", "kernel": "attn_mse", "achieved": round(mse_bytes / (mse_ms * 1e-3) / 1e9, 1),
                         "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": round(mse_bytes / (mse_ms * 1e-3) / 1e9 / pk["hbm_gbs"], 4), "traffic": None,
                         "traffic_note": "no ncu capture of this kernel",
                         "note": "the broadcast metric's kernel; the trajectory's time is the forward layer's "
                                 "(train720p / 720p lines)"},
            "e2e": None, "e2e_note": "the trajectory's inputs are produced on the device step by step in a sampler; "
                                     "no host copy belongs to a step",
            "gpu_launches": launches, "clocks": clk.summary()}
    return line


# ------------------------------------------------------------ the oracle
def oracle_sample_step(wl, sp, ctx, qblocks):
    """One bounded sample of the step on the CPU oracle: block means and scores of one
    head, selection of the sampled query blocks, their attention forward and, for
    training workloads, the backward contributions of those query blocks (their dQ and
    their shares of dK and dV for every kept key block).  Returns the algorithmic
    FLOPs of what it ran: 4 |b_i| |b_j| d per kept pair forward, 10 backward."""
    import numpy as np

    from oracle import prism_oracle as po

    Qb, Kb, Vb, dOb = ctx
    qbar = po.block_mean(Qb, wl.block)
    kbar = po.block_mean(Kb, wl.block)
    S = po.block_scores(qbar[:, qblocks], kbar)
    counts = np.zeros((1, wl.nb), np.int32)
    idx = np.zeros((1, wl.nb, wl.nb), np.int32)
    pairs = 0
    for r, i in enumerate(qblocks):
        kept, _, _ = po.select_row(S[0, r], sp, wl.cdf_tau)
        counts[0, i] = kept.size
        idx[0, i, : kept.size] = kept
        lens = np.minimum(wl.block, wl.N - kept * wl.block)
        pairs += int(lens.sum()) * min(wl.block, wl.N - i * wl.block)
    O, L = po.bsa_forward(Qb, Kb, Vb, counts, idx, wl.block, qblocks=qblocks)
    if wl.mode != "fwd+bwd":
        return 4.0 * pairs * wl.d
    po.bsa_backward(Qb, Kb, Vb, O, dOb, L, counts, idx, wl.block, qblocks=qblocks)
    return 14.0 * pairs * wl.d


def oracle_context(wl, head):
    """Head `head` of Q, K, V, dO in block order ([N, 1, d] fp64).  The block order comes
    from the oracle's zone statistics over this head's channels of V (a sample of the
    zone step, computed once, outside any timing)."""
    import numpy as np

    from audio_diffusion_dits_zone_b300 import synth
    from oracle import prism_oracle as po

    hs = [head]
    Q, K, V = (np.stack(synth.gen_heads(wl, t, hs), axis=1).astype(np.float64)
               for t in (synth.Q_ID, synth.K_ID, synth.V_ID))
    dO = np.stack(synth.gen_heads(wl, synth.DO_ID, hs), axis=1).astype(np.float64)
    _, perm, _ = po.zone_shapes([V[:, 0]], synth.gen_a2v(wl), wl.grid, wl.zone, wl.shapes)
    return Q[perm], K[perm], V[perm], dO


def cpu_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        return max(n) if n else 1
    except Exception:
        return os.cpu_count() or 1


def cpu_baseline(wl, sp, budget_s=20.0, head=0):
    """The oracle as it stands, timed on the host cores on a bounded sample."""
    ctx = oracle_context(wl, head)
    blocks = list(range(0, wl.nb, max(1, wl.nb // 64)))
    done, work, t0 = 0, 0.0, time.perf_counter()
    while done < len(blocks) and time.perf_counter() - t0 < budget_s:
        work += oracle_sample_step(wl, sp, ctx, blocks[done:done + 2])
        done += 2
    dt = time.perf_counter() - t0
    return {"value": round(work / dt / 1e12, 6), "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
            "sample": f"head {head}: block means/scores, selection and attention "
                      f"{'fwd+bwd (dQ and the dK/dV contributions of the sampled query blocks)' if wl.mode == 'fwd+bwd' else 'forward'} of {done} query blocks "
                      f"(of {wl.nb}) spread over the sequence; {dt:.1f} s of CPU time; zone statistics "
                      f"over this head's channels done once outside the timing"}


def run_pab_reference(args):
    """--impl reference for the broadcast trajectory: the oracle's rate on the 720p
    forward layer (bounded sample per step), turned into ms per denoising step for the
    trajectory's computed steps (extrapolated from the sampled work: the sampled query
    blocks' executed pairs scaled to all blocks and heads)."""
    import numpy as np

    from audio_diffusion_dits_zone_b300 import pab, synth

    wl = synth.WORKLOADS["720p"]
    ctx = oracle_context(wl, 0)
    blocks = list(range(0, wl.nb, max(1, wl.nb // 64)))
    work, dt, nblk = 0.0, 0.0, 0
    for s in range(max(1, args.steps)):
        b = blocks[(s * 2) % len(blocks):][:2]
        t0 = time.perf_counter()
        work += oracle_sample_step(wl, wl.sparsity, ctx, b)
        dt += time.perf_counter() - t0
        nblk += len(b)
    rate = work / dt  # FLOP/s of the oracle
    step_flops = work / nblk * wl.nb * wl.heads  # one computed step's forward, extrapolated
    frac = sum(pab.schedule(PAB_STEPS, PAB_RANGE)) / PAB_STEPS
    ms = frac * step_flops / rate * 1e3
    return {"metric": PAB_METRIC, "value": round(ms, 1), "unit": "ms/step", "n_gpus": args.gpus, "steps": PAB_STEPS,
            "warmup": args.warmup, "ms_per_step": round(ms, 1), "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": "pab720p (see the library's line); oracle time extrapolated from a bounded sample"},
            "cpu_baseline": {"value": round(ms, 1), "unit": "ms/step", "cores": cpu_threads(), "kind": "oracle",
                             "sample": f"{nblk} query blocks of head 0 of the 720p forward layer in {dt:.1f} s, "
                                       f"scaled to {wl.nb} blocks x {wl.heads} heads per computed step"},
            "e2e": {"value": round(ms, 1), "unit": "ms/step", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_reference(args):
    from audio_diffusion_dits_zone_b300 import synth

    if args.workload == "pab720p":
        return run_pab_reference(args)
    wl = synth.WORKLOADS[args.workload]
    sp = wl.sparsity if args.sparsity is None else args.sparsity
    ctx = oracle_context(wl, 0)
    blocks = list(range(0, wl.nb, max(1, wl.nb // 64)))
    per = 2
    for w in range(args.warmup):
        oracle_sample_step(wl, sp, ctx, blocks[(w * per) % len(blocks):][:per])
    work, t0 = 0.0, time.perf_counter()
    for s in range(args.steps):
        b = blocks[(s * per) % len(blocks):][:per]
        work += oracle_sample_step(wl, sp, ctx, b)
    dt = time.perf_counter() - t0
    v = work / dt / 1e12
    sample = (f"each step: head 0, block means/scores, selection and attention "
              f"{'fwd+bwd' if wl.mode == 'fwd+bwd' else 'forward'} of {per} query blocks "
              f"(of {wl.nb}); fp64 numpy")
    return {"metric": METRIC, "value": round(v, 6), "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(wl, sp), "impl": "reference",
            "cpu_baseline": {"value": round(v, 6), "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(v, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="train720p")
    ap.add_argument("--sparsity", type=float, default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=20.0)
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg (extra workloads)")
    ap.add_argument("--select", default="split", choices=["fused", "split"],
                    help="block scores + selection in one kernel (fused) or scores written, then selection (split)")
    ap.add_argument("--blocks", default="consecutive", choices=["consecutive", "zone-chunked"],
                    help="blocks as consecutive B-token chunks of the block order, or cut per zone")
    args = ap.parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    a2v = args.workload == "a2v720p"
    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_a2v_reference(args) if a2v else run_reference(args)), flush=True)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    run = run_a2v if a2v else (run_pab if args.workload == "pab720p" else run_ours)
    line = run(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
