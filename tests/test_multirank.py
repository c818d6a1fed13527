"""The multi-process path on the CPU (gloo, world size 2), no GPU: the bench's
reduction of a timing to the slowest rank, and the reference arm launched the
way the driver launches N > 1 (torch.distributed.run, one process per rank):
rank 0 alone measures and prints one JSON line, every rank exits 0.

The hot path itself has no collective: each rank owns its token rows of
grad_out and grad_A and a replica of the frozen NF4 weight (M-sharding), so the
ranks' kernels never wait on one another; what is shared is host logic only.
"""
from __future__ import annotations

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


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _max_worker(rank: int, world: int, port: int, out_dir: str) -> None:
    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        # Rank r took 1.5 + r milliseconds; every rank must see the slowest.
        got = bench.max_over_ranks(1.5 + rank, world, torch.device("cpu"))
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
            f.write(repr(got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gives_every_rank_the_slowest_time(tmp_path):
    world = 2
    mp.start_processes(_max_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    for r in range(world):
        assert float((tmp_path / f"rank{r}.txt").read_text()) == 2.5


def test_max_over_ranks_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(3.25, 1, torch.device("cpu")) == 3.25


def test_reference_arm_under_torchrun_prints_one_line_from_rank_0():
    pytest.importorskip("numpy")
    env = dict(os.environ, OMP_NUM_THREADS="2")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--workload", "tiny", "--steps", "2", "--warmup", "0"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    assert d["n_gpus"] == 2 and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
