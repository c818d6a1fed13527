"""bench.py's host-side bookkeeping on the CPU: the count of library kernel
launches per step that the bench line reports as gpu_launches."""
from __future__ import annotations

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from workloads import F32, Problem  # noqa: E402


def test_launches_per_step():
    w = bench.workloads(None)
    # 196 problems: 5 descriptor uploads (48 each), one streamed f16 pass, one GEMM.
    assert bench.launches_per_step(w["full_step"], "ws") == 5 + 1 + 1
    # without the ws entry: the uploads and the GEMM only
    assert bench.launches_per_step(w["full_step"], "plain") == 5 + 1
    # the MLP pair: one upload, the pass, the GEMM
    assert bench.launches_per_step(w["mlp"], "ws") == 3
    # a single problem: pre-pass and GEMM, or the plain GEMM alone
    assert bench.launches_per_step(w["q_proj"], "ws") == 2
    assert bench.launches_per_step(w["q_proj"], "plain") == 1
    # few-token problems run their own kernel, one launch each
    few = [Problem(16, 256, 256, F32, 1.0, 0.02, False, i) for i in range(3)]
    assert bench.launches_per_step(few, "ws") == 3
    assert bench.launches_per_step([few[0]], "ws") == 1
    # more problems with copies than the streamed pass takes: sequential passes
    many = [Problem(128, 64, 256, F32, 1.0, 0.02, False, i) for i in range(300)]
    assert bench.launches_per_step(many, "ws") == -(-300 // 48) + -(-300 // 64) + 1
