"""GPU parity of rms_norm_backward against the fp64 oracle (page "trueno-gpu
0.4.17 -- src/kernels/backward/rms_norm.rs", module doc).  fp32 arithmetic:
the row's dot product has H terms and dL/dgamma sums one term per row, so the
tolerance is relative to the sums of absolute values:
    |dx - ref| <= 2e-4 * (|gamma g| + |x| mean|x g gamma| / r^2) / r + 1e-30
    |dgamma - ref| <= 5e-4 * sum_rows |g x| / r + 1e-30"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from oracle import rms_norm

pytestmark = pytest.mark.gpu
EPS = 1e-6


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from backward_gemm_gb300.build import build

    build()
    import backward_gemm_gb300 as nb

    nb.lib()
    yield


def nb():
    import backward_gemm_gb300

    return backward_gemm_gb300


def _inputs(rows, H, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(rows, H, generator=g)
    gamma = 1.0 + 0.1 * torch.randn(H, generator=g)
    gy = torch.randn(rows, H, generator=g) * 1e-2
    rms = torch.sqrt((x.double() ** 2).mean(dim=1) + EPS).float()  # the forward's r, fp32
    return x, gamma, gy, rms


def _check(rows, H, seed, want_gamma=True):
    x, gamma, gy, rms = _inputs(rows, H, seed)
    dx, dgamma = nb().rms_norm_backward(x.cuda(), gamma.cuda(), rms.cuda(), gy.cuda(), want_gamma)
    nb().check_error()
    ref_dx, ref_dg, bx, bg = rms_norm.backward(x.numpy(), gamma.numpy(), rms.numpy(), gy.numpy())
    err = np.abs(dx.cpu().double().numpy() - ref_dx)
    assert (err <= 2e-4 * bx + 1e-30).all(), float((err / (bx + 1e-30)).max())
    if want_gamma:
        errg = np.abs(dgamma.cpu().double().numpy() - ref_dg)
        assert (errg <= 5e-4 * bg + 1e-30).all(), float((errg / (bg + 1e-30)).max())
    return dx, dgamma


@pytest.mark.parametrize("rows,H", [(64, 32), (7, 200), (4096, 1536), (300, 4096), (33, 8192),
                                    (1, 12), (2000, 516)])
def test_rms_norm_backward_matches_oracle(rows, H):
    _check(rows, H, seed=rows + H)


def test_rms_norm_backward_without_gamma_and_deterministic():
    a, ga = _check(1024, 1536, 5)
    b, _ = _check(1024, 1536, 5, want_gamma=False)
    assert torch.equal(a, b)  # the same per-row arithmetic with or without dL/dgamma
    c, gc = _check(1024, 1536, 5)
    assert torch.equal(a, c) and torch.equal(ga, gc)


def test_rms_norm_backward_rejects_bad_arguments():
    import ctypes as C

    L = nb().lib()
    x = torch.zeros((4, 64), device="cuda")
    p = lambda t: C.c_void_p(t.data_ptr())
    r = torch.ones(4, device="cuda")
    gm = torch.ones(64, device="cuda")
    dg = torch.empty(64, device="cuda")
    # hidden not a multiple of 4, hidden too large, no workspace for dL/dgamma
    assert L.rms_norm_backward(p(x), p(gm), p(r), p(x), p(x), None, 4, 62, None, 0, None) == 1
    assert L.rms_norm_backward(p(x), p(gm), p(r), p(x), p(x), None, 1, 8196, None, 0, None) == 1
    assert L.rms_norm_backward(p(x), p(gm), p(r), p(x), p(x), p(dg), 4, 64, None, 0, None) == 5
    # zero rows: dL/dgamma is zero
    dg.fill_(3.0)
    assert L.rms_norm_backward(None, None, None, None, None, p(dg), 0, 64, None, 0, None) == 0
    torch.cuda.synchronize()
    assert torch.all(dg == 0)
