"""Multi-process host logic of bench.py on the CPU (gloo, world size 2).

The workload shards by sequence into independent replicas (no data-path collective): the only
cross-rank steps are the barrier around the timed region and the reduction of the result, the
slowest rank's time (max) and the units of all ranks (sum).  The reference arm under torchrun
runs on rank 0 alone; the other ranks exit without work.
"""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_path):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, lr, w = bench.dist_env()
        bench.barrier(w)
        ms, units = bench.reduce_over_ranks(torch, w, 10.0 + 5.0 * rank, 100 * (rank + 1))
        bench.barrier(w)
        if rank == 0:
            with open(out_path, "w") as f:
                json.dump({"env": [r, lr, w], "ms": ms, "units": units}, f)
    finally:
        dist.destroy_process_group()


def test_reduce_over_ranks_max_time_sum_units(tmp_path):
    out = tmp_path / "rank0.json"
    mp.spawn(_rank_main, args=(2, _free_port(), str(out)), nprocs=2, join=True)
    d = json.loads(out.read_text())
    assert d["env"] == [0, 0, 2]
    assert d["ms"] == 15.0            # the slowest rank's time
    assert d["units"] == 300.0        # every rank's units
    # whole-job throughput as bench.py computes it: all units over the slowest time
    assert d["units"] / (d["ms"] / 1e3) == pytest.approx(20000.0)


def test_single_rank_needs_no_process_group():
    assert bench.reduce_over_ranks(torch, 1, 12.5, 64) == (12.5, 64)
    bench.barrier(1)


def test_reference_arm_under_torchrun_prints_once():
    """Two ranks of the reference arm on the tiny workload: one JSON line, from rank 0."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--workload", "tiny", "--gpus", "2", "--steps", "1", "--warmup", "0"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(l) for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = lines[0]
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
