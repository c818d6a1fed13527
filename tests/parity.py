"""Helpers shared by the GPU parity tests: run a problem through the C ABI and
through the oracle on the same seeded inputs, and compare.

Tolerance for grad_A (fp32 tensor-core accumulation of exact f16 products):
    |gpu - ref| <= 2e-3 * sum_n |f16(go)[m,n] * deq(B)[k,n]| + 1e-6
per element, ref = the oracle's fp64 sum.  Dequantised values and NF4 codes
are compared bit for bit.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from workloads import F32, Problem, make_grad_out, make_weight

RTOL_BOUND = 2e-3
ATOL = 1e-6


def to_device_go(go: np.ndarray, dtype: int, dev="cuda") -> torch.Tensor:
    if dtype == F32:
        return torch.from_numpy(go).to(dev)
    return torch.from_numpy(go.view(np.int16)).to(dev).view(torch.bfloat16)


def assert_close(got: np.ndarray, ref: np.ndarray, bound: np.ndarray, what: str = ""):
    got = got.astype(np.float64)
    err = np.abs(got - ref)
    tol = RTOL_BOUND * bound + ATOL
    bad = err > tol
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance; first "
            + ", ".join(f"{tuple(i)} got {got[tuple(i)]:.6g} ref {ref[tuple(i)]:.6g}" for i in idx))
    assert np.isfinite(got).all()
    return float(err.max()) if err.size else 0.0


def sample_rows(M: int, n: int = 12, seed: int = 0) -> np.ndarray:
    rng = np.random.default_rng(seed)
    fixed = {0, 1, 127, 128, M // 2, M - 2, M - 1}
    rows = sorted({r for r in fixed if 0 <= r < M} | set(rng.integers(0, M, n).tolist()))
    return np.array(rows, dtype=np.int32)


def run_problem(p: Problem, rows=None, check_codes: bool = True, entry: str = "plain"):
    """Quantise B and run the GEMM on the GPU; compare with the oracle.  rows=None
    compares every element, otherwise only the given rows of grad_A.  entry
    "ws" runs nf4_backward_a_ws (f16 pre-pass into a workspace) instead of
    nf4_backward_a_ex."""
    import backward_gemm_gb300 as nb

    go = make_grad_out(p)
    B = make_weight(p)
    w = nb.quantize(torch.from_numpy(B).cuda())
    if entry == "ws":
        ga = nb.backward_a_ws(to_device_go(go, p.go_dtype), w)
    else:
        ga = nb.backward_a(to_device_go(go, p.go_dtype), w)
    nb.check_error()
    data_o, scales_o = oracle.quantize(B)
    if check_codes:
        np.testing.assert_array_equal(w.data.cpu().numpy(), data_o)
        np.testing.assert_array_equal(w.scales.cpu().numpy(), scales_o)
    got = ga.cpu().numpy()
    if rows is None:
        ref, bound = oracle.backward_a(go, p.go_dtype, scales_o, data_o, p.K)
        return assert_close(got, ref, bound, f"{p}")
    go16 = oracle.round_operand(go, p.go_dtype)
    bt = oracle.dequantize_f16(scales_o, data_o, p.K, p.N)
    ref, bound = oracle.backward_a_rows(go16, bt, rows)
    return assert_close(got[rows], ref, bound, f"{p} rows")
