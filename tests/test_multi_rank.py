"""The N > 1 host path of bench.py on CPU with the gloo backend, world size 2:
the max-over-ranks timing and whole-job rate, and the reference arm launched
the way the driver launches it (torch.distributed.run, one process per rank:
rank 0 alone runs and prints one JSON line, the other exits 0)."""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=2)
    ms = bench.max_over_ranks([2.5, 4.0][rank], 2, "cpu")     # rank 1 is the slower one
    rate = bench.whole_job_rate(2, 1e9, ms)
    out[rank] = (ms, rate)
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_rate():
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.start_processes(_rank_main, args=(port, out), nprocs=2, start_method="spawn")
        res = dict(out)
    assert res[0] == res[1]
    ms, rate = res[0]
    assert ms == 4.0                                  # the slowest rank
    assert abs(rate - 2 * 1e9 / 4e-3 / 1e9) < 1e-9    # both ranks' work over that time: 500 GFLOP/s


def test_reference_arm_under_torchrun_world_size_2():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "1"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"
