"""Run whole steps of the path on one GPU and exit: the command that profilers wrap.

    python -m audio_diffusion_dits_zone_b300.run_step --workload 720p-4h --steps 2

Generates the workload's seeded inputs, runs `--steps` passes of zone shapes ->
pool + score -> select -> attention forward (-> backward for training workloads),
checks the device status word and prints the kernels' launch count.
"""
import argparse

import torch

from . import prism as P
from . import synth
from .pipeline import PrismLayer


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="720p-4h", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--steps", type=int, default=2)
    ap.add_argument("--sparsity", type=float, default=None)
    ap.add_argument("--select", default="split", choices=["fused", "split"])
    ap.add_argument("--blocks", default="consecutive", choices=["consecutive", "zone-chunked"])
    a = ap.parse_args()
    wl = synth.WORKLOADS[a.workload]
    layer = PrismLayer(wl, "cuda", sparsity=a.sparsity, fused_select=a.select == "fused",
                       chunked=a.blocks == "zone-chunked")
    layer.load_inputs()
    n0 = P.launch_count()
    for _ in range(a.steps):
        layer.step()
    torch.cuda.synchronize()
    w = P.status_check()
    if w:
        raise SystemExit(f"device status word 0x{w:x}")
    print(f"{a.workload}: {a.steps} steps, {P.launch_count() - n0} kernel launches, status ok")


if __name__ == "__main__":
    main()
