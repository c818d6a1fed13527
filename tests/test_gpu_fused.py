"""GPU parity of the fused sibling-projection input gradient
(nf4_backward_a_fused) against the oracle's fused sum:

    grad_x = sum_p f16(grad_out_p) @ deq(B_p)^T

over projections that read the same layer input (q/k/v, gate/up; page
"aprender-gpu 0.32.0 -- src/kernels/backward/nf4_tensor_core.rs", struct doc
comment and Qwen-dimension test).  Small cases are checked in every element,
the Qwen-shaped q/k/v and gate/up calls at M = 4096 on sampled rows; one-hot
rows must give one projection's dequantised column exactly, and the fused call
must equal the pre-converted single call on the concatenated grad_out bit for
bit.
"""
from __future__ import annotations

import ctypes as C

import numpy as np
import pytest
import torch

import oracle
from parity import assert_close, sample_rows, to_device_go
from workloads import BF16, F32, FUSED, Problem, make_grad_out, make_weight

pytestmark = pytest.mark.gpu

F16 = 2


@pytest.fixture(scope="module")
def nb():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from backward_gemm_gb300.build import build

    build()
    import backward_gemm_gb300

    backward_gemm_gb300.lib()
    return backward_gemm_gb300


def _parts(nb, probs, dtypes=None):
    """Device grad_outs, per-part weights, and the oracle's f16 operands."""
    gos, ws, go16s, bts = [], [], [], []
    for i, p in enumerate(probs):
        dt = p.go_dtype if dtypes is None else dtypes[i]
        go = make_grad_out(Problem(p.M, p.N, p.K, F32 if dt == F16 else dt, p.go_std, p.b_std,
                                   p.outliers, p.seed))
        B = make_weight(p)
        if dt == F16:
            h = oracle.f32_to_f16(go)
            gos.append(torch.from_numpy(h.view(np.int16)).cuda().view(torch.float16))
            go16s.append(h)
        else:
            gos.append(to_device_go(go, dt))
            go16s.append(oracle.round_operand(go, dt))
        ws.append(nb.quantize(torch.from_numpy(B).cuda()))
        data_o, scales_o = oracle.quantize(B)
        bts.append(oracle.dequantize_f16(scales_o, data_o, p.K, p.N))
    return gos, ws, go16s, bts


SMALL = [
    ("ragged-qkv-like", [Problem(300, 192, 640, F32, 1.0, 0.02, True, 11),
                         Problem(300, 64, 640, F32, 1.0, 0.02, False, 12),
                         Problem(300, 64, 640, F32, 1.0, 0.02, False, 13)], None),
    ("mixed-dtypes", [Problem(129, 256, 1536, BF16, 1e-2, 0.02, False, 21),
                      Problem(129, 136, 1536, F32, 1e-2, 0.02, True, 22),
                      Problem(129, 72, 1536, F32, 1.0, 0.02, False, 23)], [BF16, F32, F16]),
    ("narrow-parts", [Problem(520, 8, 384, F32, 1.0, 0.02, False, 31),
                      Problem(520, 16, 384, F32, 1.0, 0.02, False, 32),
                      Problem(520, 24, 384, BF16, 1.0, 0.02, False, 33)], None),
    ("few-tokens", [Problem(16, 1536, 1536, F32, 1e-2, 0.02, False, 41),
                    Problem(16, 256, 1536, F32, 1e-2, 0.02, False, 42)], None),
    ("one-part", [Problem(1000, 320, 256, F32, 1.0, 0.02, False, 51)], None),
]


@pytest.mark.parametrize("name,probs,dtypes", SMALL, ids=[s[0] for s in SMALL])
def test_fused_full_check_and_equals_concatenated_single_call(nb, name, probs, dtypes):
    gos, ws, go16s, bts = _parts(nb, probs, dtypes)
    w = nb.stack_weights(ws)
    got = nb.backward_a_fused(gos, w)
    again = nb.backward_a_fused(gos, w)
    nb.check_error()
    M = probs[0].M
    ref, bound = oracle.backward_a_fused_rows(go16s, bts, np.arange(M))
    assert_close(got.cpu().numpy(), ref, bound, name)
    assert torch.equal(got, again)
    # Same A operand values, same single problem: the pre-converted single call
    # on the concatenation gives the same bits (f32 widening of bf16/f16 parts
    # is exact, so their rounding to f16 is unchanged).
    cat = torch.cat([g.float() for g in gos], dim=1).contiguous()
    with nb.small_m_max(0):
        single = nb.backward_a_ws(cat, w)
    nb.check_error()
    assert torch.equal(got, single)


def test_stacked_weight_equals_quantised_concatenation(nb):
    probs = FUSED["fused_qkv"]
    Bs = [make_weight(Problem(256, p.N, p.K, F32, 1.0, p.b_std, p.outliers, p.seed))
          for p in probs]
    stacked = nb.stack_weights([nb.quantize(torch.from_numpy(B).cuda()) for B in Bs])
    whole = nb.quantize(torch.from_numpy(np.concatenate(Bs, axis=1)).cuda())
    assert torch.equal(stacked.data, whole.data) and torch.equal(stacked.scales, whole.scales)


def test_fused_one_hot_rows_recover_one_projections_columns(nb):
    Ns, K, M = (256, 64, 136), 640, 8
    ws = [nb.quantize(torch.from_numpy(make_weight(Problem(1, N, K, F32, 1.0, 0.02, True,
                                                           60 + i))).cuda())
          for i, N in enumerate(Ns)]
    picks = [(0, 0), (0, 255), (1, 63), (1, 17), (2, 0), (2, 135), (2, 64), (0, 128)]
    gos = [torch.zeros((M, N), device="cuda") for N in Ns]
    for m, (p, n) in enumerate(picks):
        gos[p][m, n] = 1.0
    got = nb.backward_a_fused(gos, nb.stack_weights(ws))
    nb.check_error()
    for m, (p, n) in enumerate(picks):
        col = nb.dequantize_f16(ws[p])[n].float()
        assert torch.equal(got[m], col), (m, p, n)


@pytest.mark.parametrize("name", sorted(FUSED))
def test_fused_qwen_shapes_sampled_rows(nb, name):
    probs = FUSED[name]
    gos, ws, go16s, bts = _parts(nb, probs)
    w = nb.stack_weights(ws)
    got = nb.backward_a_fused(gos, w)
    again = nb.backward_a_fused(gos, w)
    nb.check_error()
    rows = sample_rows(probs[0].M, 12, 7)
    ref, bound = oracle.backward_a_fused_rows(go16s, bts, rows)
    assert_close(got.cpu().numpy()[rows], ref, bound, name)
    assert torch.equal(got, again)


def test_fused_rejects_bad_arguments_without_launching(nb):
    L = nb.lib()
    M, K = 64, 128
    gos = [torch.zeros((M, 64), device="cuda"), torch.zeros((M, 64), device="cuda")]
    w = nb.stack_weights([nb.quantize(torch.zeros((K, 64), device="cuda")) for _ in gos])
    out = torch.full((M, K), 5.0, device="cuda")
    ws = nb.ws_workspace(M, 128)

    def call(parts, count=None, nbytes=None, K_=K, wsp=None):
        arr = (nb.Nf4Part * len(parts))(*[nb.Nf4Part(*x) for x in parts])
        return L.nf4_backward_a_fused(arr, len(parts) if count is None else count,
                                      C.c_void_p(w.scales.data_ptr()), C.c_void_p(w.data.data_ptr()),
                                      C.c_void_p(out.data_ptr()), M, K_,
                                      C.c_void_p(ws.data_ptr()) if wsp is None else wsp,
                                      ws.numel() if nbytes is None else nbytes, None)

    good = [(gos[0].data_ptr(), F32, 64), (gos[1].data_ptr(), F32, 64)]
    assert call([(gos[0].data_ptr(), F32, 60), good[1]]) == nb.NF4_ERR_INVALID   # N_p % 8
    assert call(good, count=0) == nb.NF4_ERR_INVALID
    assert call(good, count=65) == nb.NF4_ERR_INVALID
    assert call([(gos[0].data_ptr(), 7, 64), good[1]]) == nb.NF4_ERR_INVALID     # dtype
    assert call(good, K_=100) == nb.NF4_ERR_INVALID
    assert call([(gos[0].data_ptr() + 4, F32, 64), good[1]]) == nb.NF4_ERR_ALIGN
    assert call(good, nbytes=2 * M * 128 - 1) == nb.NF4_ERR_WORKSPACE
    assert call(good, wsp=C.c_void_p(ws.data_ptr() + 16)) == nb.NF4_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((out == 5.0).all())
    assert call(good) == nb.NF4_OK
    nb.check_error()
    assert bool((out == 0.0).all())  # zero grad_out, zero weight
    with pytest.raises(ValueError):
        nb.backward_a_fused([gos[0]], w)  # N sums to 64, the stacked weight has 128


# ---------------------------------------------------------------- grouped
def _layer_problems(nb, M, layer_seed, dtypes=None):
    """A layer's backward as fused problems: q/k/v (3 parts), o (1), gate/up
    (2), down (1), at reduced widths, with the oracle's f16 operands."""
    shapes = [((192, 64, 64), 320), ((320,), 320), ((256, 256), 320), ((320,), 512)]
    out = []
    for i, (Ns, K) in enumerate(shapes):
        probs = [Problem(M, N, K, F32, 1.0, 0.02, False, layer_seed + 10 * i + j)
                 for j, N in enumerate(Ns)]
        gos, ws, go16s, bts = _parts(nb, probs, dtypes)
        out.append((gos, nb.stack_weights(ws), go16s, bts))
    return out


def test_fused_batched_matches_single_fused_calls_and_oracle(nb):
    """Two layers' fused problems (8 problems, 14 parts) in one grouped call,
    with the pass beside the GEMM and with the pass first: both equal single
    nf4_backward_a_fused calls without a split bit for bit, and the oracle."""
    probs = _layer_problems(nb, 700, 100) + _layer_problems(nb, 700, 200, [F32, BF16, F16])
    items = [(gos, w, None) for gos, w, _, _ in probs]
    streamed = nb.backward_a_fused_batched(items)
    arr, keep, _ = nb._fused_array(items)
    r = lambda x: (x + 255) // 256 * 256
    seq_bytes = r(640 * len(items)) + sum(r(2 * gos[0].shape[0] * w.N) for gos, w, _ in items)
    ws = torch.empty(seq_bytes, dtype=torch.uint8, device="cuda")
    sequential = nb.backward_a_fused_batched(items, ws)
    nb.check_error()
    for i, ((gos, w, go16s, bts), a, b) in enumerate(zip(probs, streamed, sequential)):
        M = gos[0].shape[0]
        single = nb.backward_a_fused(gos, w, nb.ws_workspace(M, w.N, split=False))
        nb.check_error()
        assert torch.equal(a, b), f"problem {i}: streamed != sequential pass"
        assert torch.equal(a, single), f"problem {i}: grouped != single fused call"
        rows = sample_rows(M, 8, i)
        ref, bound = oracle.backward_a_fused_rows(go16s, bts, rows)
        assert_close(a.cpu().numpy()[rows], ref, bound, f"problem {i}")


def test_fused_batched_rejects_bad_problems_without_launching(nb):
    L = nb.lib()
    M, K = 300, 128
    gos = [torch.zeros((M, 64), device="cuda") for _ in range(3)]
    w = nb.stack_weights([nb.quantize(torch.zeros((K, 64), device="cuda")) for _ in gos])
    out = torch.full((M, K), 2.0, device="cuda")
    items = [(gos, w, out)]
    arr, keep, _ = nb._fused_array(items)
    need = int(L.nf4_backward_a_fused_batched_ws_bytes(arr, 1))
    assert need > 2 * M * 192
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    assert L.nf4_backward_a_fused_batched(arr, 1, None, 0, None) == nb.NF4_ERR_WORKSPACE
    keep[0][1].N = 60  # a part not a multiple of 8 columns
    assert L.nf4_backward_a_fused_batched(arr, 1, C.c_void_p(ws.data_ptr()), need, None) == \
        nb.NF4_ERR_INVALID
    keep[0][1].N = 64
    arr[0].count = 9
    assert L.nf4_backward_a_fused_batched(arr, 1, C.c_void_p(ws.data_ptr()), need, None) == \
        nb.NF4_ERR_INVALID
    torch.cuda.synchronize()
    assert bool((out == 2.0).all())
    arr[0].count = 3
    assert L.nf4_backward_a_fused_batched(arr, 1, C.c_void_p(ws.data_ptr()), need, None) == nb.NF4_OK
    nb.check_error()
    assert bool((out == 0.0).all())
