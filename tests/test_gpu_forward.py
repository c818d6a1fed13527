"""GPU parity of the forward product C[M x N] = A[M x K] @ dequant(B_nf4[K x N])
(nf4_forward_ws, the pre-converted pair kernel with a K-major B operand)
against the CPU oracle, on the same seeded inputs.  Same tolerance as the
backward: |gpu - ref| <= 2e-3 * sum_k |f16(A)[m,k] * deq(B)[k,n]| + 1e-6."""
from __future__ import annotations

import ctypes as C

import numpy as np
import pytest
import torch

import oracle
from parity import assert_close, sample_rows, to_device_go
from workloads import BF16, F32, Problem, make_grad_out, make_weight

pytestmark = pytest.mark.gpu


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


def _inputs(M, N, K, dtype, seed, a_std=1.0, b_std=0.02, outliers=False):
    """A [M, K] (fp32, or bf16 bits) and the dense weight B [K, N]."""
    a = make_grad_out(Problem(M, K, N, dtype, a_std, b_std, outliers, seed))
    B = make_weight(Problem(M, N, K, dtype, a_std, b_std, outliers, seed + 1))
    return a, B


def run_forward(M, N, K, dtype=F32, seed=0, rows=None, a_std=1.0, outliers=False,
                workspace=None):
    a, B = _inputs(M, N, K, dtype, seed, a_std, outliers=outliers)
    w = nb().quantize(torch.from_numpy(B).cuda())
    c = nb().forward_ws(to_device_go(a, dtype), w, workspace)
    nb().check_error()
    data, scales = oracle.quantize(B)
    got = c.cpu().numpy()
    if rows is None:
        ref, bound = oracle.forward(a, dtype, scales, data, N)
        assert_close(got, ref, bound, f"forward {M}x{N}x{K}")
    else:
        ref, bound = oracle.forward_rows(oracle.round_operand(a, dtype),
                                         oracle.dequantize_f16(scales, data, K, N), rows)
        assert_close(got[rows], ref, bound, f"forward {M}x{N}x{K} rows")
    return c, w, a


@pytest.mark.parametrize("M,N,K,dtype", [
    (32, 64, 128, F32),       # the tiny configuration's sizes
    (300, 520, 384, F32),     # ragged M and N (N not a multiple of the 256-column tile)
    (513, 1024, 1536, BF16),  # 3 row tiles, ragged by one row
    (1000, 772, 640, F32),
])
def test_forward_matches_oracle(M, N, K, dtype):
    run_forward(M, N, K, dtype, seed=M + N)


def test_forward_one_hot_rows_are_exact_dequantised_rows():
    """A row e_k selects row k of deq(B): C[m, :] == deq(B)[k, :] bit for bit
    (one f16 product with 1.0 per element), across NF4 blocks, stages, the two
    CTAs' column halves and the 256-column tiles."""
    M, N, K = 256, 600, 384
    ks = np.array([0, 1, 63, 64, 65, 127, 128, 191, 255, 256, 320, 383] * 21 + [5, 7, 9, 11],
                  dtype=np.int64)[:M]
    a = np.zeros((M, K), dtype=np.float32)
    a[np.arange(M), ks] = 1.0
    _, B = _inputs(M, N, K, F32, 41)
    w = nb().quantize(torch.from_numpy(B).cuda())
    c = nb().forward_ws(torch.from_numpy(a).cuda(), w)
    nb().check_error()
    deq = nb().dequantize_f16(w).float()  # [N, K]: deq(B) transposed
    want = deq[:, torch.from_numpy(ks).cuda()].T  # [M, N]
    assert torch.equal(c, want)


def test_forward_f16_input_equals_rounded_fp32_input():
    """f16 A skips the pre-pass; fp32 A rounded to f16 by the pre-pass gives the
    same operand, so the results agree bit for bit."""
    M, N, K = 640, 768, 1024
    a, B = _inputs(M, N, K, F32, 43)
    w = nb().quantize(torch.from_numpy(B).cuda())
    a32 = torch.from_numpy(a).cuda()
    c32 = nb().forward_ws(a32, w)
    c16 = nb().forward_ws(a32.half(), w)
    nb().check_error()
    assert torch.equal(c32, c16)


def test_forward_deterministic_and_tile_sizes_agree():
    """Two runs give the same bits; forced 256- and 512-token tiles sum each
    element in the same order, so they agree bit for bit too."""
    M, N, K = 2048, 1536, 1536
    a, B = _inputs(M, N, K, F32, 47, a_std=1e-2)
    w = nb().quantize(torch.from_numpy(B).cuda())
    x = torch.from_numpy(a).cuda()
    ws = nb().fwd_workspace(M, K)
    c1 = nb().forward_ws(x, w, ws)
    c2 = nb().forward_ws(x, w, ws)
    with nb().tile_rows_forced(512):
        c512 = nb().forward_ws(x, w, ws)
    with nb().tile_rows_forced(256):
        c256 = nb().forward_ws(x, w, ws)
    nb().check_error()
    assert torch.equal(c1, c2)
    assert torch.equal(c256, c512)
    data, scales = oracle.quantize(B)
    rows = sample_rows(M, 10, 47)
    ref, bound = oracle.forward_rows(oracle.round_operand(a, F32),
                                     oracle.dequantize_f16(scales, data, K, N), rows)
    assert_close(c1.cpu().numpy()[rows], ref, bound, "forward q-shaped rows")


def test_forward_split_of_last_wave_matches_oracle():
    """48 tiles of 256 x 256 with 140 stages each on 76 pairs: the last (only)
    partial wave is split by stages; results are deterministic, close to the
    unsplit run and within tolerance of the oracle."""
    M, N, K = 2048, 1536, 8960
    a, B = _inputs(M, N, K, BF16, 53, a_std=1e-2, outliers=True)
    w = nb().quantize(torch.from_numpy(B).cuda())
    x = to_device_go(a, BF16)
    with nb().tile_rows_forced(256):
        ws = nb().fwd_workspace(M, K)
        s1 = nb().forward_ws(x, w, ws)
        s2 = nb().forward_ws(x, w, ws)
        whole = nb().forward_ws(x, w, torch.empty(2 * M * K, dtype=torch.uint8, device="cuda"))
    nb().check_error()
    assert torch.equal(s1, s2)
    assert torch.allclose(s1, whole, rtol=1e-4, atol=1e-5)
    data, scales = oracle.quantize(B)
    rows = sample_rows(M, 6, 53)
    ref, bound = oracle.forward_rows(oracle.round_operand(a, BF16),
                                     oracle.dequantize_f16(scales, data, K, N), rows)
    assert_close(s1.cpu().numpy()[rows], ref, bound, "forward split rows")


def test_forward_rejects_bad_arguments_without_launching():
    L = nb().lib()
    x = torch.zeros((64, 128), device="cuda")
    w = nb().quantize(torch.zeros((128, 64), device="cuda"))
    c = torch.empty((64, 64), device="cuda")
    ws = nb().fwd_workspace(64, 128)
    p = lambda t: C.c_void_p(t.data_ptr())
    nbytes = ws.numel()
    # N % 4 != 0, K % 64 != 0, misaligned workspace, too small a workspace
    assert L.nf4_forward_ws(p(x), 0, p(w.scales), p(w.data), p(c), 64, 62, 128, p(ws), nbytes, None) == 1
    assert L.nf4_forward_ws(p(x), 0, p(w.scales), p(w.data), p(c), 64, 64, 96, p(ws), nbytes, None) == 1
    assert L.nf4_forward_ws(p(x), 0, p(w.scales), p(w.data), p(c), 64, 64, 128,
                            C.c_void_p(ws.data_ptr() + 16), nbytes - 16, None) == 5
    assert L.nf4_forward_ws(p(x), 0, p(w.scales), p(w.data), p(c), 64, 64, 128, p(ws), 1024, None) == 5
    assert L.nf4_forward_ws(p(x), 0, p(w.scales), p(w.data), p(c), 0, 64, 128, None, 0, None) == 0
    torch.cuda.synchronize()
    nb().check_error()
