"""Out-of-bounds writes: nothing is written outside grad_A (or C), or outside
the part of a workspace the call may use.

The page's kernel (page "aprender-gpu 0.32.0 -- src/kernels/backward/
nf4_tensor_core.rs", build_ptx "PHASE 4") stores whole 16 x 16 tiles and so
writes past grad_A when M or K is not a multiple of 16.  Here every store is
clipped.  Each call below writes into a view in the middle of a larger buffer
filled with a sentinel bit pattern, on ragged shapes of every path (M tails of
256- and 512-token tiles, K tails of 256-column tiles, the few-token kernel,
the forward product's N tail, stream-K splits, grouped launches); afterwards
every sentinel word before and after the view must be intact, and the view must
hold the same values as a call on a plain tensor.
"""
from __future__ import annotations

import pytest
import torch

from parity import to_device_go
from workloads import BF16, F32, Problem, make_grad_out, make_weight

pytestmark = pytest.mark.gpu

SENTINEL = -0x2A5A5A5B  # 0xD5A5A5A5 as int32: a negative NaN bit pattern
PAD = 1024              # sentinel words on each side (4 KB, keeps 16-byte alignment)


@pytest.fixture(scope="module")
def nb():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from backward_gemm_gb300.build import build

    build()
    import backward_gemm_gb300

    backward_gemm_gb300.lib()
    return backward_gemm_gb300


def guarded(rows: int, cols: int):
    """A float32 [rows, cols] view with PAD sentinel words on each side."""
    buf = torch.full((rows * cols + 2 * PAD,), SENTINEL, dtype=torch.int32, device="cuda")
    return buf, buf[PAD:PAD + rows * cols].view(torch.float32).view(rows, cols)


def assert_guards_intact(buf: torch.Tensor, n: int, what: str):
    torch.cuda.synchronize()
    head, tail = buf[:PAD], buf[PAD + n:]
    bad_h = int((head != SENTINEL).sum())
    bad_t = int((tail != SENTINEL).sum())
    assert bad_h == 0 and bad_t == 0, f"{what}: {bad_h} words before and {bad_t} after were written"


def guarded_bytes(nbytes: int):
    """A uint8 workspace of nbytes followed by 4 KB of sentinel bytes."""
    buf = torch.full((nbytes + 4 * PAD,), 0xA5, dtype=torch.uint8, device="cuda")
    return buf, buf[:nbytes]


BACKWARD = [
    Problem(8191, 1024, 4160, F32, 1.0, 0.02, False, 90, "m8191-k4160"),      # M and K tails
    Problem(1300, 2048, 4608, F32, 1.0, 0.02, False, 91, "m1300-512-tiles"),  # 512-token tail
    Problem(33, 1032, 320, BF16, 1e-2, 0.02, True, 92, "m33-bf16-k-tail"),    # few-token kernel
    Problem(300, 196, 640, F32, 1.0, 0.02, True, 93, "m300-n196"),            # N tail, pitch pad
    Problem(2560, 576, 2048, BF16, 1e-2, 0.02, True, 94, "split-wave"),       # stream-K split
    Problem(1024, 4096, 512, F32, 1.0, 0.015, True, 95, "split-512"),         # split 512-token tiles
]


@pytest.mark.parametrize("p", BACKWARD, ids=lambda p: p.name)
@pytest.mark.parametrize("entry", ["plain", "ws"])
def test_backward_writes_only_grad_a_and_its_workspace(nb, p, entry):
    go = to_device_go(make_grad_out(p), p.go_dtype)
    w = nb.quantize(torch.from_numpy(make_weight(p)).cuda())
    buf, out = guarded(p.M, p.K)
    forced = 512 if p.name in ("m1300-512-tiles", "split-512") else 0
    with nb.tile_rows_forced(forced):
        if entry == "plain":
            nb.backward_a(go, w, out=out)
            plain = nb.backward_a(go, w)
        else:
            need = int(nb.lib().nf4_backward_a_ws_bytes(p.M, p.N))
            wbuf, ws = guarded_bytes(need)
            nb.backward_a_ws(go, w, ws, out=out)
            plain = nb.backward_a_ws(go, w, nb.ws_workspace(p.M, p.N))
    nb.check_error()
    assert_guards_intact(buf, p.M * p.K, f"{p.name} {entry}: grad_A")
    if entry == "ws":
        torch.cuda.synchronize()
        assert bool((wbuf[need:] == 0xA5).all()), f"{p.name}: written past the workspace"
    assert torch.equal(out, plain)


@pytest.mark.parametrize("M,N,K", [(700, 1036, 512), (8191, 4100, 320), (64, 260, 1024)])
def test_forward_writes_only_c(nb, M, N, K):
    pa = Problem(M, K, N, F32, 1.0, 0.02, False, 96)
    a = torch.from_numpy(make_grad_out(pa)).cuda()                 # A [M, K]
    w = nb.quantize(torch.from_numpy(make_weight(Problem(M, N, K, F32, 1.0, 0.02, False, 97))).cuda())
    buf, c = guarded(M, N)
    need = int(nb.lib().nf4_forward_ws_bytes(M, K))
    wbuf, ws = guarded_bytes(need)
    nb.forward_ws(a, w, ws, out=c)
    plain = nb.forward_ws(a, w)
    nb.check_error()
    assert_guards_intact(buf, M * N, f"forward {M}x{N}x{K}: C")
    assert bool((wbuf[need:] == 0xA5).all()), "written past the workspace"
    assert torch.equal(c, plain)


@pytest.mark.parametrize("entry", ["batched", "batched_ws", "noalloc"])
def test_grouped_launches_write_only_their_outputs(nb, entry):
    probs = [BACKWARD[0], BACKWARD[2], BACKWARD[3],
             Problem(520, 136, 384, BF16, 1e-2, 0.02, False, 98, "g-bf16")]
    items, bufs, plains = [], [], []
    for p in probs:
        go = to_device_go(make_grad_out(p), p.go_dtype)
        w = nb.quantize(torch.from_numpy(make_weight(p)).cuda())
        buf, out = guarded(p.M, p.K)
        items.append((go, w, out))
        bufs.append(buf)
        plains.append(nb.backward_a(go, w))
    if entry == "batched":
        nb.backward_a_batched(items)
    elif entry == "noalloc":
        nb.backward_a_batched_noalloc(items)
    else:
        need = nb.batched_ws_bytes(items)
        wbuf, ws = guarded_bytes(need)
        nb.backward_a_batched_ws(items, ws)
        torch.cuda.synchronize()
        assert bool((wbuf[need:] == 0xA5).all()), "written past the workspace"
    nb.check_error()
    for p, buf, (_, _, out), plain in zip(probs, bufs, items, plains):
        assert_guards_intact(buf, p.M * p.K, f"{entry} {p.name}")
        assert torch.equal(out, plain), f"{entry} {p.name}"
