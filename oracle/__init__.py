"""numpy front end of the C oracle for the NF4 backward-A GEMM.

TEST INFRASTRUCTURE ONLY.  Imported by ``tests/``, by the package smoke check
and by the benchmark's CPU-baseline leg; the product path never imports it and
shares no code with it.

    grad_A[M x K] = grad_out[M x N] @ dequant(B_nf4[K x N])^T

(page "aprender-gpu 0.32.0 -- src/kernels/backward/nf4_tensor_core.rs",
struct doc comment).  Results are fp64; operands are rounded to f16 exactly as
that page's build_ptx phases 1 and 2 round them.
"""
from __future__ import annotations

import ctypes as C

import numpy as np

from . import rms_norm  # noqa: F401  (RMS layer-norm forward/backward, fp64)
from .build import build_oracle

F32 = 0
BF16 = 1

_lib = None


def lib():
    """Load (building first if needed) ``libnf4oracle.so``."""
    global _lib
    if _lib is None:
        path = build_oracle()
        L = C.CDLL(path)
        vp = C.c_void_p
        L.nf4o_codebook.argtypes = [vp]
        L.nf4o_codebook.restype = None
        L.nf4o_f32_to_f16.argtypes = [C.c_float]
        L.nf4o_f32_to_f16.restype = C.c_uint16
        L.nf4o_f32_to_f16_array.argtypes = [vp, C.c_longlong, vp]
        L.nf4o_f32_to_f16_array.restype = None
        L.nf4o_f16_to_f64.argtypes = [C.c_uint16]
        L.nf4o_f16_to_f64.restype = C.c_double
        L.nf4o_bf16_to_f32.argtypes = [C.c_uint16]
        L.nf4o_bf16_to_f32.restype = C.c_float
        L.nf4o_quantize.argtypes = [vp, C.c_int, C.c_int, vp, vp]
        L.nf4o_code_at.argtypes = [vp, C.c_int, C.c_int, C.c_int]
        L.nf4o_dequantize_f16.argtypes = [vp, vp, C.c_int, C.c_int, vp]
        L.nf4o_round_operand.argtypes = [vp, C.c_int, C.c_longlong, vp]
        L.nf4o_backward_a_rows.argtypes = [vp, vp, C.c_int, C.c_int, C.c_int, vp,
                                           C.c_int, vp, vp]
        L.nf4o_backward_a.argtypes = [vp, C.c_int, vp, vp, C.c_int, C.c_int, C.c_int,
                                      vp, vp]
        L.nf4o_backward_a_fused_rows.argtypes = [C.c_int, vp, vp, vp, C.c_int, C.c_int, vp,
                                                 C.c_int, vp, vp]
        L.nf4o_gemm_backward_b_rows.argtypes = [vp, vp, C.c_int, C.c_int, C.c_int, C.c_int, vp,
                                                C.c_int, vp, vp]
        L.nf4o_forward_rows.argtypes = [vp, vp, C.c_int, C.c_int, C.c_int, vp, C.c_int, vp, vp]
        L.nf4o_forward.argtypes = [vp, C.c_int, vp, vp, C.c_int, C.c_int, C.c_int, vp, vp]
        L.nf4o_set_threads.argtypes = [C.c_int]
        L.nf4o_set_threads.restype = None
        L.nf4o_max_threads.restype = C.c_int
        _lib = L
    return _lib


def _p(a: np.ndarray):
    return C.c_void_p(a.ctypes.data)


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (rc={rc})")


def set_threads(n: int) -> None:
    lib().nf4o_set_threads(int(n))


def max_threads() -> int:
    return int(lib().nf4o_max_threads())


def codebook() -> np.ndarray:
    out = np.zeros(16, dtype=np.float32)
    lib().nf4o_codebook(_p(out))
    return out


def f32_to_f16(x) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().nf4o_f32_to_f16_array(_p(x), x.size, _p(out))
    return out


def f16_to_f64(h) -> np.ndarray:
    h = np.asarray(h, dtype=np.uint16)
    f = lib().nf4o_f16_to_f64
    return np.array([f(int(v)) for v in h.ravel()], dtype=np.float64).reshape(h.shape)


def bf16_to_f32(b) -> np.ndarray:
    b = np.asarray(b, dtype=np.uint16)
    f = lib().nf4o_bf16_to_f32
    return np.array([f(int(v)) for v in b.ravel()], dtype=np.float32).reshape(b.shape)


def quantize(B: np.ndarray):
    """B fp32 [K, N] row-major -> (data u8 [N, K/2], scales f32 [N, K/64])."""
    B = np.ascontiguousarray(B, dtype=np.float32)
    K, N = B.shape
    data = np.zeros((N, K // 2), dtype=np.uint8)
    scales = np.zeros((N, max(K // 64, 1)), dtype=np.float32)
    _check(lib().nf4o_quantize(_p(B), K, N, _p(data), _p(scales)), "quantize")
    return data, scales


def code_at(data: np.ndarray, K: int, k: int, n: int) -> int:
    data = np.ascontiguousarray(data, dtype=np.uint8)
    return int(lib().nf4o_code_at(_p(data), K, k, n))


def dequantize_f16(scales: np.ndarray, data: np.ndarray, K: int, N: int) -> np.ndarray:
    """-> deq(B) transposed, raw f16 bits [N, K]."""
    scales = np.ascontiguousarray(scales, dtype=np.float32)
    data = np.ascontiguousarray(data, dtype=np.uint8)
    bt = np.empty((N, K), dtype=np.uint16)
    _check(lib().nf4o_dequantize_f16(_p(scales), _p(data), K, N, _p(bt)), "dequantize")
    return bt


def round_operand(go: np.ndarray, dtype: int) -> np.ndarray:
    """grad_out (fp32 array, or bf16 given as uint16 bits) -> f16 bits."""
    go = np.ascontiguousarray(go, dtype=np.float32 if dtype == F32 else np.uint16)
    out = np.empty(go.shape, dtype=np.uint16)
    _check(lib().nf4o_round_operand(_p(go), dtype, go.size, _p(out)), "round_operand")
    return out


def backward_a_rows(go16: np.ndarray, bt: np.ndarray, rows, want_bound: bool = True):
    """fp64 rows of grad_A from f16 operands: go16 [M, N], bt [N, K]."""
    go16 = np.ascontiguousarray(go16, dtype=np.uint16)
    bt = np.ascontiguousarray(bt, dtype=np.uint16)
    M, N = go16.shape
    N2, K = bt.shape
    assert N == N2
    rows = np.ascontiguousarray(rows, dtype=np.int32)
    ref = np.empty((rows.size, K), dtype=np.float64)
    bound = np.empty((rows.size, K), dtype=np.float64) if want_bound else None
    rc = lib().nf4o_backward_a_rows(_p(go16), _p(bt), M, N, K, _p(rows), rows.size,
                                    _p(ref), _p(bound) if want_bound else None)
    _check(rc, "backward_a_rows")
    return ref, bound


def backward_a(go: np.ndarray, dtype: int, scales: np.ndarray, data: np.ndarray,
               K: int, want_bound: bool = True):
    """Whole grad_A [M, K] in fp64 (and the |.|-sum bound) from raw inputs."""
    go = np.ascontiguousarray(go, dtype=np.float32 if dtype == F32 else np.uint16)
    M, N = go.shape
    scales = np.ascontiguousarray(scales, dtype=np.float32)
    data = np.ascontiguousarray(data, dtype=np.uint8)
    ref = np.empty((M, K), dtype=np.float64)
    bound = np.empty((M, K), dtype=np.float64) if want_bound else None
    rc = lib().nf4o_backward_a(_p(go), dtype, _p(scales), _p(data), M, N, K, _p(ref),
                               _p(bound) if want_bound else None)
    _check(rc, "backward_a")
    return ref, bound


def backward_a_fused_rows(go16s, bts, rows, want_bound: bool = True):
    """fp64 rows of the fused input gradient sum_p f16(go_p) @ deq(B_p)^T from
    f16 operands: go16s[p] [M, N_p], bts[p] = deq(B_p) transposed [N_p, K]."""
    go16s = [np.ascontiguousarray(g, dtype=np.uint16) for g in go16s]
    bts = [np.ascontiguousarray(b, dtype=np.uint16) for b in bts]
    P = len(go16s)
    assert P == len(bts) and P > 0
    M = go16s[0].shape[0]
    K = bts[0].shape[1]
    Ns = np.array([g.shape[1] for g in go16s], dtype=np.int32)
    for g, b in zip(go16s, bts):
        assert g.shape[0] == M and b.shape == (g.shape[1], K)
    gp = (C.c_void_p * P)(*[g.ctypes.data for g in go16s])
    bp = (C.c_void_p * P)(*[b.ctypes.data for b in bts])
    rows = np.ascontiguousarray(rows, dtype=np.int32)
    ref = np.empty((rows.size, K), dtype=np.float64)
    bound = np.empty((rows.size, K), dtype=np.float64) if want_bound else None
    rc = lib().nf4o_backward_a_fused_rows(P, gp, bp, _p(Ns), M, K, _p(rows), rows.size, _p(ref),
                                          _p(bound) if want_bound else None)
    _check(rc, "backward_a_fused_rows")
    return ref, bound


HALF_F16 = 0
HALF_BF16 = 1


def gemm_backward_b_rows(a: np.ndarray, gc: np.ndarray, dtype16: int, rows=None,
                         want_bound: bool = True):
    """fp64 rows of the dense weight gradient grad_B = A^T @ grad_C from 16-bit
    operands given as raw bits (uint16): a [M, K], gc [M, N]; dtype16 HALF_F16
    or HALF_BF16.  rows: the output rows k (default all).  Returns (ref, bound),
    each [len(rows), N]."""
    a = np.ascontiguousarray(a, dtype=np.uint16)
    gc = np.ascontiguousarray(gc, dtype=np.uint16)
    M, K = a.shape
    M2, N = gc.shape
    assert M == M2
    rows = np.arange(K, dtype=np.int32) if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
    ref = np.empty((rows.size, N), dtype=np.float64)
    bound = np.empty((rows.size, N), dtype=np.float64) if want_bound else None
    rc = lib().nf4o_gemm_backward_b_rows(_p(a), _p(gc), int(dtype16), M, K, N, _p(rows), rows.size,
                                         _p(ref), _p(bound) if want_bound else None)
    _check(rc, "gemm_backward_b_rows")
    return ref, bound


def forward_rows(a16: np.ndarray, bt: np.ndarray, rows, want_bound: bool = True):
    """fp64 rows of the forward product C = f16(A) @ deq(B) from f16 operands:
    a16 [M, K], bt = deq(B) transposed [N, K]."""
    a16 = np.ascontiguousarray(a16, dtype=np.uint16)
    bt = np.ascontiguousarray(bt, dtype=np.uint16)
    M, K = a16.shape
    N, K2 = bt.shape
    assert K == K2
    rows = np.ascontiguousarray(rows, dtype=np.int32)
    ref = np.empty((rows.size, N), dtype=np.float64)
    bound = np.empty((rows.size, N), dtype=np.float64) if want_bound else None
    rc = lib().nf4o_forward_rows(_p(a16), _p(bt), M, N, K, _p(rows), rows.size, _p(ref),
                                 _p(bound) if want_bound else None)
    _check(rc, "forward_rows")
    return ref, bound


def forward(a: np.ndarray, dtype: int, scales: np.ndarray, data: np.ndarray, N: int,
            want_bound: bool = True):
    """Whole forward product C [M, N] = f16(A)[M, K] @ deq(B)[K, N] in fp64
    (and the |.|-sum bound) from raw inputs (A fp32, or bf16 as uint16 bits)."""
    a = np.ascontiguousarray(a, dtype=np.float32 if dtype == F32 else np.uint16)
    M, K = a.shape
    scales = np.ascontiguousarray(scales, dtype=np.float32)
    data = np.ascontiguousarray(data, dtype=np.uint8)
    ref = np.empty((M, N), dtype=np.float64)
    bound = np.empty((M, N), dtype=np.float64) if want_bound else None
    rc = lib().nf4o_forward(_p(a), dtype, _p(scales), _p(data), M, N, K, _p(ref),
                            _p(bound) if want_bound else None)
    _check(rc, "forward")
    return ref, bound
