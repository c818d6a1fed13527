"""The grouped backward-A entry point that allocates nothing.

Callers that cannot allocate device memory (inside a caching allocator they
must not re-enter, in a stream-ordered region where cudaMalloc would
synchronise, or with all device memory reserved up front) use
nf4_backward_a_batched_noalloc, which keeps its descriptors in a fixed array
inside the library.  It promises the same problems, rules and results as
nf4_backward_a_batched, so every output is compared with that entry point's bit
for bit, and with the oracle within the tolerance of every parity test.

This file is collected last on purpose, so that a run that stops at the first
failure has run every other test first; it also passes when run alone in a
fresh process.
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


def _inputs(nb, problems):
    """Device inputs and the oracle's whole grad_A (and bound) per problem."""
    items, refs = [], []
    for p in problems:
        go = make_grad_out(p)
        B = make_weight(p)
        items.append((to_device_go(go, p.go_dtype), nb.quantize(torch.from_numpy(B).cuda())))
        data_o, scales_o = oracle.quantize(B)
        refs.append(oracle.backward_a(go, p.go_dtype, scales_o, data_o, p.K))
    return items, refs


def _noalloc_call(nb, items, outs):
    """One call of the entry point through the C ABI."""
    arr = (nb.Nf4Problem * len(items))()
    for i, ((go, w), out) in enumerate(zip(items, outs)):
        M, N = go.shape
        arr[i] = nb.Nf4Problem(go.data_ptr(), nb.NF4_F32 if go.dtype == torch.float32
                               else nb.NF4_BF16, w.scales.data_ptr(), w.data.data_ptr(),
                               out.data_ptr(), M, N, w.K)
    stream = torch.cuda.current_stream().cuda_stream
    rc = nb.lib().nf4_backward_a_batched_noalloc(arr, len(items), C.c_void_p(stream))
    assert rc == nb.NF4_OK, nb.status_string(rc)
    nb.check_error()


def _check_two_calls(nb, problems):
    items, refs = _inputs(nb, problems)
    # Output of the existing grouped entry point (caller-owned workspace).
    grouped = nb.backward_a_batched([(go, w, None) for go, w in items])
    nb.check_error()
    for call in range(2):
        # NaN-filled outputs: every element must be written by this call.
        outs = [torch.full_like(g, float("nan")) for g in grouped]
        _noalloc_call(nb, items, outs)
        for p, g, o, (ref, bound) in zip(problems, grouped, outs, refs):
            assert torch.equal(o, g), f"call {call} {p}: differs from nf4_backward_a_batched"
            assert_close(o.cpu().numpy(), ref, bound, f"call {call} {p}")


def test_noalloc_matches_grouped_entry_point_and_oracle_on_two_calls(nb):
    _check_two_calls(nb, PROBLEMS)


def _many(count: int, seed0: int) -> list[Problem]:
    """`count` small problems of varied shapes (M above the few-token limit,
    ragged tiles, fp32 and bf16 grad_out)."""
    rng = np.random.default_rng(seed0)
    out = []
    for i in range(count):
        M = int(rng.integers(65, 300))
        N = int(rng.choice([64, 72, 136, 256]))
        K = int(rng.choice([64, 128, 320]))
        dt = BF16 if i % 3 == 1 else F32
        out.append(Problem(M, N, K, dt, 1.0 if dt == F32 else 1e-2, 0.02, False, seed0 + i))
    return out


def test_noalloc_second_descriptor_upload_chunk(nb):
    """60 problems: the descriptors of problems 48 and on go up in a second
    upload, written further into the library's array."""
    _check_two_calls(nb, _many(60, 1000))


def test_noalloc_exactly_as_many_problems_as_the_array_holds(nb):
    _check_two_calls(nb, _many(256, 2000))


def test_noalloc_rejects_more_problems_than_its_array_holds(nb):
    L = nb.lib()
    arr = (nb.Nf4Problem * 257)()
    rc = L.nf4_backward_a_batched_noalloc(arr, 257, None)
    assert rc == nb.NF4_ERR_WORKSPACE
