"""The grouped backward-A entry point that allocates nothing.

Callers that cannot allocate device memory (inside a caching allocator they
must not re-enter, in a stream-ordered region where cudaMalloc would
synchronise, or with all device memory reserved up front) use
nf4_backward_a_batched_noalloc, which keeps its descriptors in a fixed array
inside the library.  This file is collected last on purpose, so that a run that
stops at the first failure has run every other test first; it also passes when
run alone in a fresh process.
"""
from __future__ import annotations

import ctypes as C

import numpy as np
import pytest
import torch

import oracle
from parity import assert_close, to_device_go
from workloads import BF16, F32, Problem, make_grad_out, make_weight

pytestmark = pytest.mark.gpu

PROBLEMS = [Problem(300, 192, 640, F32, 1.0, 0.02, True, 41),
            Problem(129, 256, 1536, BF16, 1e-2, 0.02, False, 42),
            Problem(64, 72, 64, F32, 1e-2, 0.02, False, 43),
            Problem(1000, 64, 256, F32, 1.0, 0.02, False, 44)]


@pytest.fixture(scope="module")
def nb():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from backward_gemm_gb300.build import build

    build()
    import backward_gemm_gb300

    backward_gemm_gb300.lib()
    return backward_gemm_gb300


def _inputs(nb):
    items, bounds = [], []
    for p in PROBLEMS:
        go = make_grad_out(p)
        B = make_weight(p)
        items.append((to_device_go(go, p.go_dtype), nb.quantize(torch.from_numpy(B).cuda())))
        data_o, scales_o = oracle.quantize(B)
        bounds.append(oracle.backward_a(go, p.go_dtype, scales_o, data_o, p.K)[1])
    return items, bounds


def test_noalloc_matches_grouped_entry_point_on_two_calls(nb):
    items, bounds = _inputs(nb)
    # Output of the existing grouped entry point (caller-owned workspace).
    ref = nb.backward_a_batched([(go, w, None) for go, w in items])
    nb.check_error()
    L = nb.lib()
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        outs = [torch.full_like(r, float("nan")) for r in ref]
        arr = (nb.Nf4Problem * len(items))()
        for i, ((go, w), out) in enumerate(zip(items, outs)):
            M, N = go.shape
            arr[i] = nb.Nf4Problem(go.data_ptr(), nb.NF4_F32 if go.dtype == torch.float32
                                   else nb.NF4_BF16, w.scales.data_ptr(), w.data.data_ptr(),
                                   out.data_ptr(), M, N, w.K)
        rc = L.nf4_backward_a_batched_noalloc(arr, len(items), C.c_void_p(stream))
        assert rc == nb.NF4_OK, nb.status_string(rc)
        nb.check_error()
        for p, r, o, bound in zip(PROBLEMS, ref, outs, bounds):
            # Same tolerance as every parity test, with the existing entry
            # point's result in place of the oracle's.
            assert_close(o.cpu().numpy(), r.cpu().numpy().astype(np.float64), bound,
                         f"call {call} {p}")


def test_noalloc_rejects_more_problems_than_its_array_holds(nb):
    L = nb.lib()
    arr = (nb.Nf4Problem * 257)()
    rc = L.nf4_backward_a_batched_noalloc(arr, 257, None)
    assert rc == nb.NF4_ERR_WORKSPACE
