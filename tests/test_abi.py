"""The C ABI (no GPU needed): the library builds, loads, exports every function
that include/nf4bwd.h declares, and rejects bad arguments on the host before
touching the device."""
from __future__ import annotations

import ctypes as C
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nf4bwd.h")


@pytest.fixture(scope="module")
def lib():
    from backward_gemm_gb300.build import build

    build()
    import backward_gemm_gb300 as nb

    return nb.lib()


def declared_functions() -> list[str]:
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b((?:nf4|rms_norm)_\w+)\s*\(", text)))


def test_header_declares_the_documented_calls():
    names = declared_functions()
    for n in ("nf4_quantize", "nf4_dequantize_f16", "nf4_backward_a", "nf4_backward_a_ex",
              "nf4_backward_a_batched", "nf4_backward_a_batched_workspace", "nf4_check_error",
              "nf4_status_string", "nf4_abi_version", "nf4_forward_ws", "nf4_forward_ws_bytes",
              "rms_norm_backward", "rms_norm_backward_ws_bytes"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", lib._name], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT ((?:nf4|rms_norm)_\w+)", out))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    for n in declared_functions():
        assert getattr(lib, n) is not None


def test_binding_covers_every_declared_symbol():
    import backward_gemm_gb300 as nb

    assert set(declared_functions()) <= set(nb.SIGNATURES)


def test_status_strings(lib):
    import backward_gemm_gb300 as nb

    assert lib.nf4_abi_version() == 1
    assert nb.status_string(nb.NF4_OK) == "ok"
    assert "timed out" in nb.status_string(nb.NF4_ERR_TIMEOUT)
    assert nb.status_string(99) == "unknown status"


def test_host_validation_rejects_before_any_device_work(lib):
    import backward_gemm_gb300 as nb

    fake = C.c_void_p(0x100000)  # never dereferenced: every call below fails validation
    # K not a multiple of 64, negative sizes, unknown dtype, null pointers.
    assert lib.nf4_backward_a(fake, fake, fake, fake, 16, 64, 100, None) == nb.NF4_ERR_INVALID
    assert lib.nf4_backward_a(fake, fake, fake, fake, -1, 64, 128, None) == nb.NF4_ERR_INVALID
    assert lib.nf4_backward_a_ex(fake, 7, fake, fake, fake, 16, 64, 128, None) == nb.NF4_ERR_INVALID
    assert lib.nf4_backward_a(None, fake, fake, fake, 16, 64, 128, None) == nb.NF4_ERR_INVALID
    # N not a multiple of the TMA row alignment (4 fp32 / 8 bf16 elements).
    assert lib.nf4_backward_a(fake, fake, fake, fake, 16, 66, 128, None) == nb.NF4_ERR_INVALID
    assert lib.nf4_backward_a_ex(fake, nb.NF4_BF16, fake, fake, fake, 16, 68, 128,
                                 None) == nb.NF4_ERR_INVALID
    # Misaligned pointers.
    odd = C.c_void_p(0x100004)
    assert lib.nf4_backward_a(odd, fake, fake, fake, 16, 64, 128, None) == nb.NF4_ERR_ALIGN
    assert lib.nf4_backward_a(fake, fake, fake, odd, 16, 64, 128, None) == nb.NF4_ERR_ALIGN
    assert lib.nf4_quantize(fake, 100, 8, fake, fake, None) == nb.NF4_ERR_INVALID
    assert lib.nf4_dequantize_f16(fake, fake, 96, 8, fake, None) == nb.NF4_ERR_INVALID
    # Grouped launch: a bad count or a bad problem is rejected.
    assert lib.nf4_backward_a_batched(None, -1, None, 0, None) == nb.NF4_ERR_INVALID
    probs = (nb.Nf4Problem * 1)(nb.Nf4Problem(0x100000, 0, 0x100000, 0x100000, 0x100000,
                                              16, 64, 100))
    assert lib.nf4_backward_a_batched(probs, 1, None, 0, None) == nb.NF4_ERR_INVALID
    assert lib.nf4_backward_a_batched_workspace(196) >= 196 * 384
    assert lib.nf4_backward_a_batched_workspace(0) == 0


def test_empty_problems_enqueue_nothing(lib):
    import backward_gemm_gb300 as nb

    fake = C.c_void_p(0x100000)
    # M == 0 is a no-op that needs no valid pointers (nothing is read or written).
    assert lib.nf4_backward_a(None, None, None, None, 0, 64, 128, None) == nb.NF4_OK
    assert lib.nf4_backward_a_batched(None, 0, None, 0, None) == nb.NF4_OK


def test_forward_and_rms_norm_validation_before_any_device_work(lib):
    import backward_gemm_gb300 as nb

    fake = C.c_void_p(0x100000)  # never dereferenced: every call below fails validation
    odd = C.c_void_p(0x100004)
    # Forward: K % 64, N % 4, unknown dtype, null and misaligned pointers, workspace.
    assert lib.nf4_forward_ws(fake, 0, fake, fake, fake, 16, 64, 100, fake, 1 << 20,
                              None) == nb.NF4_ERR_INVALID
    assert lib.nf4_forward_ws(fake, 0, fake, fake, fake, 16, 66, 128, fake, 1 << 20,
                              None) == nb.NF4_ERR_INVALID
    assert lib.nf4_forward_ws(fake, 9, fake, fake, fake, 16, 64, 128, fake, 1 << 20,
                              None) == nb.NF4_ERR_INVALID
    assert lib.nf4_forward_ws(None, 0, fake, fake, fake, 16, 64, 128, fake, 1 << 20,
                              None) == nb.NF4_ERR_INVALID
    assert lib.nf4_forward_ws(odd, 0, fake, fake, fake, 16, 64, 128, fake, 1 << 20,
                              None) == nb.NF4_ERR_ALIGN
    assert lib.nf4_forward_ws(fake, 0, fake, fake, fake, 16, 64, 128, None, 0,
                              None) == nb.NF4_ERR_WORKSPACE
    assert lib.nf4_forward_ws(None, 0, None, None, None, 0, 64, 128, None, 0, None) == nb.NF4_OK
    # RMSNorm backward: hidden % 4, hidden > 8192, negative rows, pointers, workspace.
    assert lib.rms_norm_backward(fake, fake, fake, fake, fake, None, 4, 62, None, 0,
                                 None) == nb.NF4_ERR_INVALID
    assert lib.rms_norm_backward(fake, fake, fake, fake, fake, None, 4, 8196, None, 0,
                                 None) == nb.NF4_ERR_INVALID
    assert lib.rms_norm_backward(fake, fake, fake, fake, fake, None, -1, 64, None, 0,
                                 None) == nb.NF4_ERR_INVALID
    assert lib.rms_norm_backward(None, fake, fake, fake, fake, None, 4, 64, None, 0,
                                 None) == nb.NF4_ERR_INVALID
    assert lib.rms_norm_backward(odd, fake, fake, fake, fake, None, 4, 64, None, 0,
                                 None) == nb.NF4_ERR_ALIGN
    assert lib.rms_norm_backward(fake, fake, fake, fake, fake, fake, 4, 64, None, 0,
                                 None) == nb.NF4_ERR_WORKSPACE


def test_grouped_bindings_check_every_item_before_any_launch(monkeypatch):
    """The grouped bindings apply the single-call rules to every item (N equal to
    the weight's, out float32 [M, K], the weight's codes and scales of the right
    size) and raise before the library is called or anything is allocated."""
    import torch

    import backward_gemm_gb300 as nb

    def no_library():
        raise AssertionError("the library was reached")

    monkeypatch.setattr(nb, "lib", no_library)
    M, N, K = 100, 64, 128
    w = nb.NF4Weight(torch.zeros((N, K // 2), dtype=torch.uint8), torch.zeros((N, K // 64)), K, N)
    go = torch.zeros((M, N))
    good_out = torch.zeros((M, K))
    cases = {
        "out too small": (go, w, torch.zeros((M, K - 64))),
        "out not float32": (go, w, torch.zeros((M, K), dtype=torch.float16)),
        "N differs from the weight's": (torch.zeros((M, N + 8)), w, good_out),
        "codes of the wrong size": (go, nb.NF4Weight(torch.zeros((N, K // 4), dtype=torch.uint8),
                                                     w.scales, K, N), good_out),
        "scales of the wrong size": (go, nb.NF4Weight(w.data, torch.zeros((N, 1)), K, N), good_out),
        "grad_out not 2-D": (torch.zeros((M, N, 1)), w, good_out),
    }
    for what, bad in cases.items():
        for call in (nb.backward_a_batched, nb.backward_a_batched_ws, nb.backward_a_batched_noalloc):
            with pytest.raises(ValueError):
                call([(go, w, good_out), bad])
        with pytest.raises(ValueError):
            nb.backward_a(bad[0], bad[1], bad[2])
    # A well-formed item still needs CUDA tensors: refused on the host as well.
    with pytest.raises(ValueError, match="CUDA"):
        nb.backward_a_batched([(go, w, good_out)])
    # The no-allocation call never creates outputs.
    with pytest.raises(ValueError):
        nb.backward_a_batched_noalloc([(go, w, None)])
