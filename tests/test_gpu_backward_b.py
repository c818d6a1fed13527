"""GPU parity of the dense weight gradient grad_B = A^T @ grad_C
(nf4_gemm_backward_b; page "trueno-gpu 0.4.17 -- src/kernels/backward/mod.rs",
GemmBackwardBKernel) against the oracle's fp64 sum over tokens, at the
tolerance of every parity test: |gpu - ref| <= 2e-3 * sum_m |a * g| + 1e-6.
"""
from __future__ import annotations

import ctypes as C

import numpy as np
import pytest
import torch

import oracle
from parity import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def nb():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from backward_gemm_gb300.build import build

    build()
    import backward_gemm_gb300

    backward_gemm_gb300.lib()
    return backward_gemm_gb300


def _inputs(M, K, N, dt, seed, a_std=0.5, c_std=0.01):
    g = torch.Generator().manual_seed(seed)
    a = (torch.randn(M, K, generator=g) * a_std).to(dt)
    c = (torch.randn(M, N, generator=g) * c_std).to(dt)
    bits = lambda t: t.view(torch.int16).numpy().view(np.uint16)
    d16 = oracle.HALF_BF16 if dt == torch.bfloat16 else oracle.HALF_F16
    return a, c, bits(a), bits(c), d16


CASES = [  # M tokens, K rows, N columns
    (300, 136, 200, torch.bfloat16, "ragged-all"),
    (64, 256, 256, torch.float16, "one-stage-one-tile"),
    (1000, 520, 264, torch.bfloat16, "tails-past-tiles"),
    (4096, 16, 1032, torch.bfloat16, "lora-rank-16"),
    (129, 1024, 1024, torch.float16, "many-tiles"),
]


@pytest.mark.parametrize("M,K,N,dt,name", CASES, ids=[c[-1] for c in CASES])
def test_backward_b_full_check(nb, M, K, N, dt, name):
    a, c, ab, cb, d16 = _inputs(M, K, N, dt, M + K + N)
    got = nb.gemm_backward_b(a.cuda(), c.cuda())
    again = nb.gemm_backward_b(a.cuda(), c.cuda())
    nb.check_error()
    ref, bound = oracle.gemm_backward_b_rows(ab, cb, d16)
    assert_close(got.cpu().numpy(), ref, bound, name)
    assert torch.equal(got, again)


def test_backward_b_split_and_unsplit_agree(nb):
    """Few output tiles and many tokens: the call splits the tokens (fp32
    partial sums added in split order); without a workspace it does not.  Both
    match the oracle; the split result is repeatable."""
    M, K, N = 8192, 256, 512
    L = nb.lib()
    assert int(L.nf4_gemm_backward_b_splits(M, K, N, 76)) > 1
    assert int(L.nf4_gemm_backward_b_ws_bytes(M, K, N)) > 0
    a, c, ab, cb, d16 = _inputs(M, K, N, torch.bfloat16, 7)
    ad, cd = a.cuda(), c.cuda()
    split = nb.gemm_backward_b(ad, cd)
    split2 = nb.gemm_backward_b(ad, cd)
    whole = nb.gemm_backward_b(ad, cd, workspace=torch.empty(256, dtype=torch.uint8, device="cuda"))
    nb.check_error()
    ref, bound = oracle.gemm_backward_b_rows(ab, cb, d16)
    assert_close(split.cpu().numpy(), ref, bound, "split")
    assert_close(whole.cpu().numpy(), ref, bound, "unsplit")
    assert torch.equal(split, split2)
    # Same products, summed in another order: equal up to rounding, but not all
    # bits (this checks that the split took place).
    assert not torch.equal(split, whole)


def test_backward_b_one_hot_tokens_pick_rows_exactly(nb):
    M, K, N = 200, 264, 136
    _, c, _, cb, _ = _inputs(M, K, N, torch.bfloat16, 3)
    a = torch.zeros((M, K), dtype=torch.bfloat16)
    picks = {0: 5, 17: 199, 255: 64, 256: 0, 263: 130}  # k -> token m
    for k, m in picks.items():
        a[m, k] = 1.0
    got = nb.gemm_backward_b(a.cuda(), c.cuda())
    nb.check_error()
    cf = c.float()
    for k in range(K):
        want = cf[picks[k]] if k in picks else torch.zeros(N)
        assert torch.equal(got[k].cpu(), want), k


def test_backward_b_rejects_bad_arguments_without_launching(nb):
    L = nb.lib()
    a = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    c = torch.zeros((64, 64), dtype=torch.bfloat16, device="cuda")
    out = torch.full((64, 64), 3.0, device="cuda")
    P = lambda t, off=0: C.c_void_p(t.data_ptr() + off)
    assert L.nf4_gemm_backward_b(P(a), P(c), 0, P(out), 64, 64, 64, None, 0, None) == nb.NF4_ERR_INVALID
    assert L.nf4_gemm_backward_b(P(a), P(c), 1, P(out), 64, 60, 64, None, 0, None) == nb.NF4_ERR_INVALID
    assert L.nf4_gemm_backward_b(P(a), P(c), 1, P(out), 64, 64, 12, None, 0, None) == nb.NF4_ERR_INVALID
    assert L.nf4_gemm_backward_b(P(a, 2), P(c), 1, P(out), 64, 64, 64, None, 0, None) == nb.NF4_ERR_ALIGN
    assert L.nf4_gemm_backward_b(P(a), P(c), 1, P(out, 4), 64, 64, 64, None, 0, None) == nb.NF4_ERR_ALIGN
    torch.cuda.synchronize()
    assert bool((out == 3.0).all())
    assert L.nf4_gemm_backward_b(None, None, 1, P(out), 0, 64, 64, None, 0, None) == nb.NF4_OK
    nb.check_error()
    assert bool((out == 0.0).all())
