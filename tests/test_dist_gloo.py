"""The multi-rank logic of bench.py on CPU: two gloo ranks, each timing its own replica,
agree on the slowest rank's time and on the whole-job throughput."""
import os
import socket

import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [120.0, 87.5][rank]
        worst = bench.max_over_ranks(local_ms, "cpu")
        out[rank] = (worst, bench.job_throughput(1e12, world, worst * 1e-3))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    port = _free_port()
    out = mp.Manager().dict()
    mp.spawn(_rank, args=(2, port, out), nprocs=2, join=True)
    assert out[0] == out[1]
    worst, tput = out[0]
    assert worst == 120.0
    assert abs(tput - 2 * 1e12 / 0.120 / 1e12) < 1e-9


def test_reference_arm_under_two_ranks_prints_one_line():
    # launched the way a multi-GPU run is launched: rank 0 alone runs the oracle and prints;
    # the other rank exits 0 without work
    import json
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py", "--impl", "reference",
           "--workload", "720p", "--steps", "1", "--warmup", "0"]
    r = subprocess.run(cmd, cwd=root, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    assert lines[0]["impl"] == "reference" and lines[0]["value"] > 0
