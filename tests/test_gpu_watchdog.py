"""The bounded waits' failure path, on a GPU, without a GPU fault.

Every wait in the library's kernels gives up after a limit, records a timeout
and where it happened in the library's status word, and lets the kernel
return.  A self-test kernel makes a wait run out on purpose (an mbarrier that
nothing arrives on, a short limit); the host then reads the status and its
site through nf4_check_error_site, the status is cleared by that read, and the
context stays usable for a normal GEMM afterwards.
"""
from __future__ import annotations

import ctypes as C

import numpy as np
import pytest
import torch

import oracle
from parity import assert_close
from workloads import CONFIGS, make_grad_out, make_weight

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


def test_wait_gives_up_reports_its_site_and_the_context_survives(nb):
    L = nb.lib()
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert L.nf4_check_error(stream) == nb.NF4_OK  # nothing pending from earlier tests
    where = nb.watchdog_selftest(200_000)
    site = (C.c_uint * 4)()
    assert L.nf4_check_error_site(stream, site) == nb.NF4_ERR_TIMEOUT
    w = where.cpu().numpy().view(np.uint32)
    assert w[1] == 0, "the wait on a barrier nobody arrives on reported success"
    assert w[2] == 0, "the second wait did not stop on the abort flag"
    assert tuple(site) == (1, 0, int(w[0]), 0)  # block 0 (+1), thread 0, the barrier, parity 0
    # The read cleared the status: the next check is clean.
    assert L.nf4_check_error_site(stream, site) == nb.NF4_OK
    assert tuple(site) == (0, 0, 0, 0)
    # The context is intact: a normal call gives the oracle's result.
    p = CONFIGS["tiny"][0]
    go, B = make_grad_out(p), make_weight(p)
    got = nb.backward_a(torch.from_numpy(go).cuda(), nb.quantize(torch.from_numpy(B).cuda()))
    nb.check_error()
    data_o, scales_o = oracle.quantize(B)
    ref, bound = oracle.backward_a(go, p.go_dtype, scales_o, data_o, p.K)
    assert_close(got.cpu().numpy(), ref, bound, "after a timeout")


def test_python_check_error_raises_with_the_site(nb):
    nb.watchdog_selftest(100_000)
    with pytest.raises(nb.Nf4Error, match="block 0, thread 0"):
        nb.check_error()
    nb.check_error()  # cleared


def test_selftest_rejects_bad_limits(nb):
    L = nb.lib()
    where = torch.zeros(3, dtype=torch.int32, device="cuda")
    p = C.c_void_p(where.data_ptr())
    assert L.nf4_watchdog_selftest(10, p, None) == nb.NF4_ERR_INVALID
    assert L.nf4_watchdog_selftest(3_000_000_000, p, None) == nb.NF4_ERR_INVALID
    assert L.nf4_watchdog_selftest(100_000, None, None) == nb.NF4_ERR_INVALID
    torch.cuda.synchronize()
    assert L.nf4_check_error(None) == nb.NF4_OK
