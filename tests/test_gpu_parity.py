"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle.

Ordered from the most diagnostic to the broadest: codes and dequantised
operands bit for bit, GEMMs whose exact answer isolates one operand's layout
(one-hot grad_out rows, an identity weight), then seeded problems that span
several tiles with ragged tails, the grouped launch, and the full-size
workloads on sampled rows.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from parity import assert_close, run_problem, sample_rows, to_device_go
from workloads import BF16, CONFIGS, F32, Problem, make_grad_out, make_weight

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


# ---------------------------------------------------------------- quantise / dequantise
@pytest.mark.parametrize("K,N,outliers,std", [(128, 64, False, 0.02), (1536, 256, True, 0.02),
                                             (640, 72, False, 1.0), (64, 4, True, 0.015)])
def test_quantize_codes_bit_exact(K, N, outliers, std):
    B = make_weight(Problem(1, N, K, F32, 1.0, std, outliers, seed=K + N))
    B[:64, :2] = 0.0  # all-zero blocks
    w = nb().quantize(torch.from_numpy(B).cuda())
    data_o, scales_o = oracle.quantize(B)
    np.testing.assert_array_equal(w.scales.cpu().numpy(), scales_o)
    np.testing.assert_array_equal(w.data.cpu().numpy(), data_o)


@pytest.mark.parametrize("K,N", [(128, 64), (1536, 256), (640, 72)])
def test_dequantize_bit_exact(K, N):
    B = make_weight(Problem(1, N, K, F32, 1.0, 0.02, True, seed=3 * K + N))
    data_o, scales_o = oracle.quantize(B)
    w = nb().NF4Weight(torch.from_numpy(data_o).cuda(), torch.from_numpy(scales_o).cuda(), K, N)
    bt = nb().dequantize_f16(w).cpu().view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(bt, oracle.dequantize_f16(scales_o, data_o, K, N))


# ---------------------------------------------------------------- exact-answer GEMMs
def _weight_from_oracle(B):
    data_o, scales_o = oracle.quantize(B)
    w = nb().NF4Weight(torch.from_numpy(data_o).cuda(), torch.from_numpy(scales_o).cuda(),
                       B.shape[0], B.shape[1])
    return w, data_o, scales_o


def test_one_hot_rows_give_dequantised_columns_exactly():
    """go[m, :] = e_n  =>  grad_A[m, :] = deq(B)[:, n] exactly (one product by 1.0)."""
    K, N = 640, 192
    B = make_weight(Problem(1, N, K, F32, 1.0, 0.02, True, seed=5))
    w, data_o, scales_o = _weight_from_oracle(B)
    ns = [0, 1, 7, 8, 15, 16, 63, 64, 65, 127, 128, 191]
    M = 2 * len(ns) + 130  # rows in two M tiles, the rest zero
    go = np.zeros((M, N), dtype=np.float32)
    for i, n in enumerate(ns):
        go[i, n] = 1.0
        go[129 + i, n] = 1.0
    ga = nb().backward_a(torch.from_numpy(go).cuda(), w).cpu().numpy()
    bt = oracle.dequantize_f16(scales_o, data_o, K, N).view(np.float16).astype(np.float32)
    for i, n in enumerate(ns):
        np.testing.assert_array_equal(ga[i], bt[n], err_msg=f"row {i} n={n}")
        np.testing.assert_array_equal(ga[129 + i], bt[n], err_msg=f"row {129 + i} n={n}")
    assert np.all(ga[len(ns):129] == 0) and np.all(ga[129 + len(ns):] == 0)


@pytest.mark.parametrize("dtype", [F32, BF16])
def test_identity_weight_returns_rounded_grad_out(dtype):
    """B = I (K = N): deq(B) is exactly I, so grad_A = f16(grad_out) exactly."""
    K = N = 320
    B = np.eye(K, N, dtype=np.float32)
    w, _, _ = _weight_from_oracle(B)
    p = Problem(200, N, K, dtype, 1.0, seed=9)
    go = make_grad_out(p)
    ga = nb().backward_a(to_device_go(go, dtype), w).cpu().numpy()
    want = oracle.round_operand(go, dtype).view(np.float16).astype(np.float32)
    np.testing.assert_array_equal(ga, want)


# ---------------------------------------------------------------- seeded problems
SMALL = [
    Problem(32, 64, 128, F32, 1.0, 0.02, False, 0, "tiny"),
    Problem(300, 192, 640, F32, 1.0, 0.02, True, 1, "ragged-3x3"),
    Problem(129, 72, 64, F32, 1e-2, 0.02, False, 2, "n-tail"),
    Problem(257, 136, 384, BF16, 1e-2, 0.02, True, 3, "bf16-ragged"),
    Problem(17, 4, 256, F32, 1.0, 0.02, False, 4, "n4"),
    Problem(5, 8, 192, BF16, 1.0, 0.02, False, 5, "n8-bf16"),
    Problem(2048, 128, 4096, F32, 1.0, 0.015, False, 6, "persistent-256-tiles"),
]


@pytest.mark.parametrize("p", SMALL, ids=lambda p: p.name)
def test_small_problems_full_check(p):
    run_problem(p)


# ---------------------------------------------------------------- few-token path
# M <= 64 runs the swap-AB kernel with N split over a cluster; the same
# problems also run through the general kernel (small-M limit 0).
FEW = [
    Problem(1, 64, 64, F32, 1.0, 0.02, False, 20, "m1-k64"),
    Problem(16, 1536, 1536, F32, 1e-2, 0.02, False, 21, "m16-q"),
    Problem(16, 200, 320, F32, 1.0, 0.02, True, 22, "m16-ragged"),
    Problem(13, 4104, 192, BF16, 1.0, 0.02, True, 23, "m13-bf16-long-n"),
    Problem(32, 520, 640, F32, 1.0, 0.02, False, 24, "m32"),
    Problem(17, 1032, 384, BF16, 1e-2, 0.02, True, 25, "m17-bf16"),
    Problem(64, 2048, 256, F32, 1.0, 0.015, False, 26, "m64"),
    Problem(33, 96, 1088, BF16, 1.0, 0.02, False, 27, "m33-bf16-k-tail"),
    Problem(16, 14336, 256, F32, 1.0, 0.015, False, 28, "m16-max-split"),
]


@pytest.mark.parametrize("route", ["few-token", "general"])
@pytest.mark.parametrize("p", FEW, ids=lambda p: p.name)
def test_few_token_problems_full_check(p, route):
    with nb().small_m_max(64 if route == "few-token" else 0):
        run_problem(p)


def test_few_token_one_hot_rows_exact():
    """One-hot rows on the split path: exactly one cluster rank holds the
    nonzero product, the other partials are zeros, so the sum is exact."""
    K, N = 384, 1280
    B = make_weight(Problem(1, N, K, F32, 1.0, 0.02, True, seed=29))
    w, data_o, scales_o = _weight_from_oracle(B)
    ns = [0, 63, 64, 127, 128, 639, 640, 641, 1000, 1279]
    go = np.zeros((len(ns) + 2, N), dtype=np.float32)
    for i, n in enumerate(ns):
        go[i, n] = 1.0
    with nb().small_m_max(64):
        ga = nb().backward_a(torch.from_numpy(go).cuda(), w).cpu().numpy()
    bt = oracle.dequantize_f16(scales_o, data_o, K, N).view(np.float16).astype(np.float32)
    for i, n in enumerate(ns):
        np.testing.assert_array_equal(ga[i], bt[n], err_msg=f"row {i} n={n}")
    assert np.all(ga[len(ns):] == 0)


def test_few_token_deterministic():
    p = Problem(16, 14336, 1024, F32, 1.0, 0.015, False, 30)
    go = to_device_go(make_grad_out(p), F32)
    w = nb().quantize(torch.from_numpy(make_weight(p)).cuda())
    with nb().small_m_max(64):
        a = nb().backward_a(go, w)
        for _ in range(3):
            assert torch.equal(a, nb().backward_a(go, w))
    nb().check_error()


def test_deterministic():
    p = Problem(300, 192, 640, F32, 1.0, 0.02, True, 11)
    go = to_device_go(make_grad_out(p), F32)
    w = nb().quantize(torch.from_numpy(make_weight(p)).cuda())
    a = nb().backward_a(go, w)
    b = nb().backward_a(go, w)
    assert torch.equal(a, b)


@pytest.mark.parametrize("name", ["down_proj", "large_a", "q_proj", "small_m_a", "small_m_b"])
def test_full_size_runs_are_bit_identical(name):
    """Three launches on the same inputs give the same grad_A in every element:
    no float atomics, no split reductions, and no race between the pipeline's
    roles can change a result."""
    p = {q.name: q for ps in CONFIGS.values() for q in ps}[name]
    go = to_device_go(make_grad_out(p), p.go_dtype)
    w = nb().quantize(torch.from_numpy(make_weight(p)).cuda())
    first = nb().backward_a(go, w)
    for _ in range(2):
        again = nb().backward_a(go, w)
        nb().check_error()
        assert torch.equal(first, again), name


def test_batched_matches_single_and_oracle():
    probs = [Problem(300, 192, 640, F32, 1.0, 0.02, True, 21),
             Problem(129, 256, 1536, BF16, 1e-2, 0.02, False, 22),
             Problem(64, 72, 64, F32, 1e-2, 0.02, False, 23),
             Problem(1000, 64, 256, F32, 1.0, 0.02, False, 24)]
    items, gos, ws, Bs = [], [], [], []
    for p in probs:
        go = make_grad_out(p)
        B = make_weight(p)
        w = nb().quantize(torch.from_numpy(B).cuda())
        items.append((to_device_go(go, p.go_dtype), w, None))
        gos.append(go)
        Bs.append(B)
        ws.append(w)
    outs = nb().backward_a_batched(items)
    nb().check_error()
    for p, go, B, (go_t, w, _), out in zip(probs, gos, Bs, items, outs):
        single = nb().backward_a(go_t, w)
        assert torch.equal(out, single), p
        data_o, scales_o = oracle.quantize(B)
        ref, bound = oracle.backward_a(go, p.go_dtype, scales_o, data_o, p.K)
        assert_close(out.cpu().numpy(), ref, bound, str(p))


def test_grouped_full_step_repeated_launches_are_identical():
    """The 196-projection training step as one grouped launch, 12 times: no wait
    may give up and every launch must give the same grad_A bit for bit.  (A
    raw-ring slot shared by both converter groups once let a parity wait pass
    on stale data: wrong values first, then a stall, after a few such launches.)"""
    probs = CONFIGS["full_step"]
    g = torch.Generator(device="cuda")
    g.manual_seed(7)
    items = []
    for p in probs:
        go = torch.randn((p.M, p.N), device="cuda", generator=g) * p.go_std
        w = nb().NF4Weight(torch.randint(0, 256, (p.N, p.K // 2), dtype=torch.uint8, device="cuda",
                                         generator=g),
                           torch.rand((p.N, p.K // 64), device="cuda", generator=g) * 0.05, p.K, p.N)
        items.append((go, w, torch.empty((p.M, p.K), device="cuda")))
    ws = nb().batched_workspace(len(items))
    watch = [0, 5, 6, 98, 195]  # q, up, down of layer 0; a middle and the last projection
    first = None
    for _ in range(12):
        outs = nb().backward_a_batched(items, ws)
        nb().check_error()
        snap = [outs[i].clone() for i in watch]
        if first is None:
            first = snap
        else:
            for i, a, b in zip(watch, first, snap):
                assert torch.equal(a, b), f"projection {i} differs between launches"
    del items, outs, first


def test_batched_bf16_only_matches_single():
    """A grouped launch whose problems all have bf16 grad_out (the deeper-ring
    layout) gives the single-problem results bit for bit."""
    probs = [Problem(300, 136, 640, BF16, 1e-2, 0.02, True, 51),
             Problem(520, 512, 1536, BF16, 1e-2, 0.02, False, 52)]
    items = [(to_device_go(make_grad_out(p), p.go_dtype),
              nb().quantize(torch.from_numpy(make_weight(p)).cuda()), None) for p in probs]
    outs = nb().backward_a_batched(items)
    nb().check_error()
    for (go, w, _), out in zip(items, outs):
        assert torch.equal(out, nb().backward_a(go, w))


def test_batched_full_step_shapes_one_layer():
    """One layer's seven projections at a reduced token count, grouped."""
    full = CONFIGS["full_step"][:7]
    probs = [Problem(256, p.N, p.K, p.go_dtype, p.go_std, p.b_std, p.outliers, p.seed, p.name)
             for p in full]
    items, refs = [], []
    for p in probs:
        go = make_grad_out(p)
        B = make_weight(p)
        items.append((to_device_go(go, p.go_dtype), nb().quantize(torch.from_numpy(B).cuda()), None))
        data_o, scales_o = oracle.quantize(B)
        go16 = oracle.round_operand(go, p.go_dtype)
        bt = oracle.dequantize_f16(scales_o, data_o, p.K, p.N)
        rows = sample_rows(p.M, 6, p.seed)
        refs.append((rows,) + oracle.backward_a_rows(go16, bt, rows))
    outs = nb().backward_a_batched(items)
    nb().check_error()
    for p, out, (rows, ref, bound) in zip(probs, outs, refs):
        assert_close(out.cpu().numpy()[rows], ref, bound, p.name)


def test_batched_call_captured_in_cuda_graph():
    """The grouped launch's descriptors travel by value, so a captured call replays
    correctly after everything the host built for it is gone."""
    import gc

    probs = [Problem(300, 192, 640, F32, 1.0, 0.02, True, 31),
             Problem(129, 256, 1536, BF16, 1e-2, 0.02, False, 32)]
    items = [(to_device_go(make_grad_out(p), p.go_dtype),
              nb().quantize(torch.from_numpy(make_weight(p)).cuda()), None) for p in probs]
    eager = nb().backward_a_batched(items)
    outs = [torch.zeros_like(e) for e in eager]
    ws = nb().batched_workspace(len(items))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        nb().backward_a_batched([(go, w, o) for (go, w, _), o in zip(items, outs)], ws)
    gc.collect()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    nb().check_error()
    for e, o in zip(eager, outs):
        assert torch.equal(e, o)


# ---------------------------------------------------------------- edge cases
def test_empty_and_degenerate():
    w = nb().quantize(torch.from_numpy(make_weight(Problem(1, 64, 128))).cuda())
    out = nb().backward_a(torch.zeros((0, 64), device="cuda"), w)
    assert out.shape == (0, 128)
    # N == 0: empty sum, grad_A is zero.
    w0 = nb().NF4Weight(torch.zeros((0, 64), dtype=torch.uint8, device="cuda"),
                        torch.zeros((0, 2), device="cuda"), 128, 0)
    out = torch.full((3, 128), 7.0, device="cuda")
    nb().backward_a(torch.zeros((3, 0), device="cuda"), w0, out=out)
    torch.cuda.synchronize()
    assert torch.all(out == 0)
    # grad_out all zero gives zeros.
    out = nb().backward_a(torch.zeros((40, 64), device="cuda"), w)
    assert torch.all(out == 0)


def test_rejects_bad_arguments_without_launching():
    L = nb().lib()
    go = torch.zeros((16, 64), device="cuda")
    w = nb().quantize(torch.from_numpy(make_weight(Problem(1, 64, 128))).cuda())
    out = torch.zeros((16, 128), device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    args = lambda **kw: [kw.get("go", go.data_ptr()), w.scales.data_ptr(), w.data.data_ptr(),
                         kw.get("out", out.data_ptr()), 16, kw.get("N", 64), kw.get("K", 128), s]
    assert L.nf4_backward_a(*args(K=100)) == nb().NF4_ERR_INVALID
    assert L.nf4_backward_a(*args(N=66)) == nb().NF4_ERR_INVALID
    assert L.nf4_backward_a(*args(go=go.data_ptr() + 4)) == nb().NF4_ERR_ALIGN
    assert L.nf4_backward_a(*args(out=out.data_ptr() + 8)) == nb().NF4_ERR_ALIGN
    assert L.nf4_backward_a(*args(go=None)) == nb().NF4_ERR_INVALID
    # Grouped launch without (or with too small) a workspace.
    go100 = torch.zeros((100, 64), device="cuda")
    out100 = torch.zeros((100, 128), device="cuda")
    probs = (nb().Nf4Problem * 1)(nb().Nf4Problem(go100.data_ptr(), 0, w.scales.data_ptr(),
                                                  w.data.data_ptr(), out100.data_ptr(), 100, 64,
                                                  128))
    assert L.nf4_backward_a_batched(probs, 1, None, 0, s) == nb().NF4_ERR_WORKSPACE
    ws = torch.empty(64, dtype=torch.uint8, device="cuda")
    assert L.nf4_backward_a_batched(probs, 1, ws.data_ptr(), 64, s) == nb().NF4_ERR_WORKSPACE
    # Few-token problems run as their own launches and need no workspace.
    few = (nb().Nf4Problem * 1)(nb().Nf4Problem(go.data_ptr(), 0, w.scales.data_ptr(),
                                                w.data.data_ptr(), out.data_ptr(), 16, 64, 128))
    out.fill_(1.0)
    assert L.nf4_backward_a_batched(few, 1, None, 0, s) == nb().NF4_OK
    nb().check_error()
    assert torch.all(out == 0)  # grad_out is zero


# ---------------------------------------------------------------- full-size workloads
FULL = [(name, p) for name in ("q_proj", "mlp", "large") for p in CONFIGS[name]]


@pytest.mark.parametrize("name,p", FULL, ids=[p.name for _, p in FULL])
def test_full_size_sampled_rows(name, p):
    run_problem(p, rows=sample_rows(p.M, 10, p.seed))


# ---------------------------------------------------------------- pre-converted entry point
# nf4_backward_a_ws rounds grad_out to f16 in a pass of its own and feeds the
# GEMM's A operand by TMA.  With a workspace that holds only the f16 copy, the
# tiles, the MMAs and their order are those of the plain entry point, so the
# two results agree bit for bit; with the full workspace a last partial wave of
# tiles is split by stages over all pairs (nf4_split_plan) and the partial sums
# are added in pair order.
WS = SMALL + [
    Problem(300, 196, 640, F32, 1.0, 0.02, True, 40, "ws-pitch-pad"),   # f16 rows padded to 200
    Problem(200, 4, 192, F32, 1.0, 0.02, False, 41, "ws-n4"),            # one half group per row
    Problem(513, 1032, 768, BF16, 1e-2, 0.02, True, 42, "ws-bf16-3-row-pairs"),
    Problem(512, 4096, 512, F32, 1e-2, 0.015, False, 44, "ws-4-tiles-of-64-stages"),  # ~19 pairs a tile
    Problem(2560, 576, 2048, BF16, 1e-2, 0.02, True, 45, "ws-80-tiles"),  # one wave + 4 split tiles
]


@pytest.mark.parametrize("p", WS, ids=lambda p: p.name)
def test_ws_full_check(p):
    with nb().small_m_max(0):
        run_problem(p, entry="ws")


@pytest.mark.parametrize("p", WS, ids=lambda p: p.name)
def test_ws_unsplit_equals_plain_bitwise(p):
    go = to_device_go(make_grad_out(p), p.go_dtype)
    w = nb().quantize(torch.from_numpy(make_weight(p)).cuda())
    with nb().small_m_max(0):
        plain = nb().backward_a(go, w)
        pre = nb().backward_a_ws(go, w, nb().ws_workspace(p.M, p.N, split=False))
    nb().check_error()
    assert torch.equal(plain, pre)


def test_ws_split_is_deterministic_and_close_to_unsplit():
    p = Problem(512, 4096, 512, F32, 1.0, 0.015, True, 46)
    go = to_device_go(make_grad_out(p), p.go_dtype)
    w = nb().quantize(torch.from_numpy(make_weight(p)).cuda())
    ws = nb().ws_workspace(p.M, p.N)
    runs = [nb().backward_a_ws(go, w, ws) for _ in range(3)]
    whole = nb().backward_a_ws(go, w, nb().ws_workspace(p.M, p.N, split=False))
    nb().check_error()
    assert torch.equal(runs[0], runs[1]) and torch.equal(runs[0], runs[2])
    # Same products, different fp32 summation order: equal up to rounding.
    assert torch.allclose(runs[0], whole, rtol=1e-4, atol=1e-4)
    # 4 tiles of 64 stages over every pair: each tile is split many ways, so
    # some element rounds differently (this checks the split took place).
    assert not torch.equal(runs[0], whole)


def test_ws_whole_waves_plus_split_wave_sampled_rows():
    """96 tiles of 64 stages on a 152-SM GB300 (76 pairs): one whole wave, then
    20 tiles split by stages over all pairs (some pairs finish a split tile and
    also wrote a partial sum for another)."""
    p = Problem(2048, 4096, 3072, BF16, 1e-2, 0.02, True, 47, "ws-96-tiles")
    run_problem(p, rows=sample_rows(p.M, 8, p.seed), check_codes=False, entry="ws")
    go = to_device_go(make_grad_out(p), p.go_dtype)
    w = nb().quantize(torch.from_numpy(make_weight(p)).cuda())
    ws = nb().ws_workspace(p.M, p.N)
    a = nb().backward_a_ws(go, w, ws)
    b = nb().backward_a_ws(go, w, ws)
    whole = nb().backward_a_ws(go, w, nb().ws_workspace(p.M, p.N, split=False))
    nb().check_error()
    assert torch.equal(a, b)
    assert torch.allclose(a, whole, rtol=1e-4, atol=1e-5)


@pytest.mark.parametrize("name,p", FULL, ids=[p.name for _, p in FULL])
def test_ws_full_size_sampled_rows_and_deterministic(name, p):
    if p.M <= 64:
        pytest.skip("few-token shapes take the same path through both entry points")
    run_problem(p, rows=sample_rows(p.M, 6, p.seed + 1), check_codes=False, entry="ws")
    go = to_device_go(make_grad_out(p), p.go_dtype)
    w = nb().quantize(torch.from_numpy(make_weight(p)).cuda())
    ws = nb().ws_workspace(p.M, p.N)
    first = nb().backward_a_ws(go, w, ws)
    again = nb().backward_a_ws(go, w, ws)
    unsplit = nb().backward_a_ws(go, w, nb().ws_workspace(p.M, p.N, split=False))
    plain = nb().backward_a(go, w)
    nb().check_error()
    assert torch.equal(first, again)
    assert torch.equal(unsplit, plain)


def test_ws_rejects_bad_workspace_without_launching():
    import ctypes as C

    L = nb().lib()
    p = Problem(300, 192, 640, F32, 1.0, 0.02, False, 43)
    go = to_device_go(make_grad_out(p), F32)
    w = nb().quantize(torch.from_numpy(make_weight(p)).cuda())
    need = int(L.nf4_backward_a_ws_bytes(p.M, p.N))
    copy = 2 * p.M * ((p.N + 7) // 8 * 8)  # the f16 copy alone
    assert need >= copy + 256 * 1024       # plus the split's flags and partial sums
    out = torch.full((p.M, p.K), 7.0, device="cuda")
    ws = torch.empty(need + 512, dtype=torch.uint8, device="cuda")

    def call(ptr, nbytes, M=p.M):
        return L.nf4_backward_a_ws(C.c_void_p(go.data_ptr()), F32, C.c_void_p(w.scales.data_ptr()),
                                   C.c_void_p(w.data.data_ptr()), C.c_void_p(out.data_ptr()), M,
                                   p.N, p.K, ptr, nbytes, None)

    with nb().small_m_max(64):
        assert call(None, 0) == nb().NF4_ERR_WORKSPACE
        assert call(C.c_void_p(ws.data_ptr()), copy - 1) == nb().NF4_ERR_WORKSPACE
        assert call(C.c_void_p(ws.data_ptr() + 16), need) == nb().NF4_ERR_WORKSPACE
        torch.cuda.synchronize()
        assert bool((out == 7.0).all())
        # Few tokens: the few-token kernel, no workspace needed.
        assert call(None, 0, M=16) == nb().NF4_OK
        nb().check_error()
        assert call(C.c_void_p(ws.data_ptr()), need) == nb().NF4_OK
        nb().check_error()
        assert call(C.c_void_p(ws.data_ptr()), copy) == nb().NF4_OK  # no room to split: whole tiles
        nb().check_error()


# ---------------------------------------------------------------- f16 grad_out
# grad_out given in f16 is the A operand as is: the oracle's operand-level
# product (f16 operands, exact products, fp64 sum) is the reference, and the
# result equals that of the same values given in fp32 through the unsplit
# pre-converted path (the conversion to f16 is then exact).
F16_CASES = [
    Problem(300, 200, 640, F32, 1.0, 0.02, True, 50, "f16-ragged"),
    Problem(16, 1536, 1536, F32, 1e-2, 0.02, False, 51, "f16-m16"),
    Problem(600, 4096, 512, F32, 1e-2, 0.015, False, 52, "f16-long-n"),
]


@pytest.mark.parametrize("p", F16_CASES, ids=lambda p: p.name)
def test_f16_grad_out_matches_oracle_and_f32_path(p):
    go32 = make_grad_out(p)
    go16 = oracle.f32_to_f16(go32)                      # f16 bits, RNE
    B = make_weight(p)
    w = nb().quantize(torch.from_numpy(B).cuda())
    go_dev = torch.from_numpy(go16.view(np.int16)).cuda().view(torch.float16)
    got = nb().backward_a(go_dev, w)
    nb().check_error()
    data_o, scales_o = oracle.quantize(B)
    bt = oracle.dequantize_f16(scales_o, data_o, p.K, p.N)
    ref, bound = oracle.backward_a_rows(go16, bt, np.arange(p.M, dtype=np.int32))
    assert_close(got.cpu().numpy(), ref, bound, f"{p}")
    # The same values in fp32 (exactly representable) through the pre-pass.
    go_back = torch.from_numpy(go16.view(np.float16).astype(np.float32)).cuda()
    with nb().small_m_max(0):
        via32 = nb().backward_a_ws(go_back, w, nb().ws_workspace(p.M, p.N, split=False))
    nb().check_error()
    assert torch.equal(got, via32)


def test_f16_grad_out_rejected_by_grouped_launch():
    p = Problem(300, 192, 640, F32, 1.0, 0.02, False, 53)
    w = nb().quantize(torch.from_numpy(make_weight(p)).cuda())
    go = torch.zeros((p.M, p.N), dtype=torch.float16, device="cuda")
    with pytest.raises(nb().Nf4Error):
        nb().backward_a_batched([(go, w, None)])


# ---------------------------------------------------------------- grouped, pre-converted
def test_batched_ws_matches_single_ws_and_oracle():
    """nf4_backward_a_batched_ws: one f16 copy per fp32/bf16 problem, f16 input
    read in place, few-token problems on their own kernel; every result equals
    the single pre-converted call without a split (or the few-token call) bit
    for bit, and the oracle within tolerance."""
    probs = [Problem(300, 192, 640, F32, 1.0, 0.02, True, 61),
             Problem(129, 256, 1536, BF16, 1e-2, 0.02, False, 62),
             Problem(16, 1536, 1536, F32, 1e-2, 0.02, False, 63),     # few tokens
             Problem(1000, 64, 256, F32, 1.0, 0.02, False, 64),
             Problem(520, 196, 384, F32, 1.0, 0.02, True, 65)]        # f16 rows padded
    items, gos, Bs = [], [], []
    for p in probs:
        go = make_grad_out(p)
        B = make_weight(p)
        items.append((to_device_go(go, p.go_dtype), nb().quantize(torch.from_numpy(B).cuda()), None))
        gos.append(go)
        Bs.append(B)
    # One more problem given in f16 (read in place).
    pf = Problem(400, 320, 512, F32, 1.0, 0.02, False, 66)
    go16 = oracle.f32_to_f16(make_grad_out(pf))
    Bf = make_weight(pf)
    items.append((torch.from_numpy(go16.view(np.int16)).cuda().view(torch.float16),
                  nb().quantize(torch.from_numpy(Bf).cuda()), None))
    outs = nb().backward_a_batched_ws(items)
    nb().check_error()
    for p, go, B, (go_t, w, _), out in zip(probs, gos, Bs, items, outs):
        single = nb().backward_a_ws(go_t, w, nb().ws_workspace(p.M, p.N, split=False))
        assert torch.equal(out, single), p
        data_o, scales_o = oracle.quantize(B)
        ref, bound = oracle.backward_a(go, p.go_dtype, scales_o, data_o, p.K)
        assert_close(out.cpu().numpy(), ref, bound, str(p))
    go_t, w, _ = items[-1]
    assert torch.equal(outs[-1], nb().backward_a(go_t, w))
    data_o, scales_o = oracle.quantize(Bf)
    bt = oracle.dequantize_f16(scales_o, data_o, pf.K, pf.N)
    ref, bound = oracle.backward_a_rows(go16, bt, np.arange(pf.M, dtype=np.int32))
    assert_close(outs[-1].cpu().numpy(), ref, bound, "f16 input")


def test_batched_ws_full_step_one_layer_and_repeatable():
    full = CONFIGS["full_step"][:7]
    probs = [Problem(512, p.N, p.K, p.go_dtype, p.go_std, p.b_std, p.outliers, p.seed, p.name)
             for p in full]
    items, refs = [], []
    for p in probs:
        go = make_grad_out(p)
        B = make_weight(p)
        items.append((to_device_go(go, p.go_dtype), nb().quantize(torch.from_numpy(B).cuda()), None))
        data_o, scales_o = oracle.quantize(B)
        go16 = oracle.round_operand(go, p.go_dtype)
        bt = oracle.dequantize_f16(scales_o, data_o, p.K, p.N)
        rows = sample_rows(p.M, 6, p.seed)
        refs.append((rows,) + oracle.backward_a_rows(go16, bt, rows))
    ws = nb().batched_ws_workspace(items)
    outs = nb().backward_a_batched_ws(items, ws)
    again = nb().backward_a_batched_ws([(g, w, None) for g, w, _ in items], ws)
    nb().check_error()
    for p, out, out2, (rows, ref, bound) in zip(probs, outs, again, refs):
        assert_close(out.cpu().numpy()[rows], ref, bound, p.name)
        assert torch.equal(out, out2)


def test_batched_ws_rejects_small_workspace_without_launching():
    import ctypes as C

    p = Problem(300, 192, 640, F32, 1.0, 0.02, False, 67)
    go = to_device_go(make_grad_out(p), F32)
    w = nb().quantize(torch.from_numpy(make_weight(p)).cuda())
    out = torch.full((p.M, p.K), 3.0, device="cuda")
    items = [(go, w, out)]
    need = nb().batched_ws_bytes(items)
    assert need >= 2 * p.M * p.N
    arr = (nb().Nf4Problem * 1)()
    arr[0] = nb().Nf4Problem(go.data_ptr(), F32, w.scales.data_ptr(), w.data.data_ptr(),
                             out.data_ptr(), p.M, p.N, p.K)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    L = nb().lib()
    # Below the descriptors and the f16 copies: rejected.  (Between that and
    # `need`, the f16 pass runs before the GEMM instead of beside it.)
    least = _sequential_ws_bytes(items)
    assert least < need
    assert L.nf4_backward_a_batched_ws(arr, 1, C.c_void_p(ws.data_ptr()), least - 1, None) == \
        nb().NF4_ERR_WORKSPACE
    assert L.nf4_backward_a_batched_ws(arr, 1, None, 0, None) == nb().NF4_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((out == 3.0).all())
    assert L.nf4_backward_a_batched_ws(arr, 1, C.c_void_p(ws.data_ptr()), need, None) == nb().NF4_OK
    nb().check_error()
    assert L.nf4_backward_a_batched_ws(arr, 1, C.c_void_p(ws.data_ptr()), least, None) == nb().NF4_OK
    nb().check_error()


# ---------------------------------------------------------------- 512-token pair tiles
# The pre-converted kernel's second variant issues two M = 256 MMA blocks per
# dequantised B^T stage.  Each output element still sums the same products in
# the same stage and K-step order, so the result equals the 256-token kernel's.
@pytest.mark.parametrize("dtype", [F32, BF16])
def test_ws_512_token_tiles_match_plain_and_oracle(dtype):
    p = Problem(2048, 4096, 4096, dtype, 1e-2, 0.015, True, 70 + dtype, "ws-512-rows")
    assert nb().tile_rows(p.M, p.N, p.K, 76) == 512
    run_problem(p, rows=sample_rows(p.M, 8, p.seed), check_codes=False, entry="ws")
    go = to_device_go(make_grad_out(p), p.go_dtype)
    w = nb().quantize(torch.from_numpy(make_weight(p)).cuda())
    a = nb().backward_a_ws(go, w)
    b = nb().backward_a_ws(go, w)
    plain = nb().backward_a(go, w)
    nb().check_error()
    assert torch.equal(a, b)
    assert torch.equal(a, plain)


def test_ws_512_token_tiles_ragged_rows():
    """M = 1300: the last 512-token tile has 276 rows, its second M-block only
    20 (TMA zero fill above M, stores clipped)."""
    p = Problem(1300, 2048, 4608, F32, 1.0, 0.02, False, 72, "ws-512-ragged")
    run_problem(p, rows=sample_rows(p.M, 10, p.seed), check_codes=False, entry="ws")
    go = to_device_go(make_grad_out(p), p.go_dtype)
    w = nb().quantize(torch.from_numpy(make_weight(p)).cuda())
    assert torch.equal(nb().backward_a_ws(go, w), nb().backward_a(go, w))
    nb().check_error()


@pytest.mark.parametrize("p", [Problem(512, 64, 256, F32, 1.0, 0.02, False, 73, "one-512-tile"),
                               Problem(700, 136, 768, BF16, 1.0, 0.02, True, 74, "ragged-512"),
                               Problem(300, 4, 192, F32, 1.0, 0.02, False, 75, "n4-512")],
                         ids=lambda p: p.name)
def test_forced_512_token_tiles_equal_256_and_oracle(p):
    go = to_device_go(make_grad_out(p), p.go_dtype)
    w = nb().quantize(torch.from_numpy(make_weight(p)).cuda())
    with nb().tile_rows_forced(512), nb().small_m_max(0):
        a = nb().backward_a_ws(go, w, nb().ws_workspace(p.M, p.N, split=False))
        run_problem(p, entry="ws")
    with nb().tile_rows_forced(256), nb().small_m_max(0):
        b = nb().backward_a_ws(go, w, nb().ws_workspace(p.M, p.N, split=False))
    nb().check_error()
    assert torch.equal(a, b)


# ---------------------------------------------------------------- split with 512-token tiles
def test_split_with_512_token_tiles_matches_oracle_and_is_deterministic():
    """4 tiles of 512 x 256 and 64 stages over every pair: each tile split ~19
    ways, partial sums of both M-blocks added in pair order."""
    p = Problem(1024, 4096, 512, F32, 1.0, 0.015, True, 80, "split-512")
    with nb().tile_rows_forced(512):
        run_problem(p, entry="ws")
        go = to_device_go(make_grad_out(p), p.go_dtype)
        w = nb().quantize(torch.from_numpy(make_weight(p)).cuda())
        ws = nb().ws_workspace(p.M, p.N)
        a = nb().backward_a_ws(go, w, ws)
        b = nb().backward_a_ws(go, w, ws)
        whole = nb().backward_a_ws(go, w, nb().ws_workspace(p.M, p.N, split=False))
    nb().check_error()
    assert torch.equal(a, b)
    assert torch.allclose(a, whole, rtol=1e-4, atol=1e-4)
    assert not torch.equal(a, whole)  # the split took place


def test_whole_waves_plus_split_wave_with_512_token_tiles():
    """90 tiles of 512 x 256 on a 152-SM GB300 (76 pairs): one whole wave, then
    14 tiles split over all pairs."""
    p = Problem(5120, 4096, 2304, BF16, 1e-2, 0.02, True, 81, "split-512-mixed")
    with nb().tile_rows_forced(512):
        run_problem(p, rows=sample_rows(p.M, 8, p.seed), check_codes=False, entry="ws")
        go = to_device_go(make_grad_out(p), p.go_dtype)
        w = nb().quantize(torch.from_numpy(make_weight(p)).cuda())
        ws = nb().ws_workspace(p.M, p.N)
        a = nb().backward_a_ws(go, w, ws)
        b = nb().backward_a_ws(go, w, ws)
        whole = nb().backward_a_ws(go, w, nb().ws_workspace(p.M, p.N, split=False))
    nb().check_error()
    assert torch.equal(a, b)
    assert torch.allclose(a, whole, rtol=1e-4, atol=1e-5)


def _sequential_ws_bytes(items) -> int:
    """Workspace of nf4_backward_a_batched_ws with no room for the streamed
    pass's bookkeeping: the descriptors and the f16 copies only."""
    r = lambda x: (x + 255) // 256 * 256
    n = r(640 * len(items))
    for go, w, _ in items:
        M, N = go.shape
        if M > 0 and N > 0 and go.dtype != torch.float16:
            n += r(2 * M * ((N + 7) // 8 * 8))
    return n


def test_batched_ws_streamed_and_sequential_passes_agree():
    """With room for its bookkeeping, the grouped pre-converted launch runs its
    f16 pass beside the GEMM (the GEMM waits per 256-row block); without, the
    pass runs first.  Both give the same bits, and the oracle's values."""
    probs = [Problem(1300, 2048, 1536, F32, 1e-2, 0.02, False, 91),   # ragged 512-row tail
             Problem(300, 136, 640, BF16, 1e-2, 0.02, True, 92),
             Problem(16, 512, 256, F32, 1.0, 0.02, False, 93),        # few tokens
             Problem(4096, 256, 1536, F32, 1e-2, 0.02, False, 94),
             Problem(513, 1032, 768, F32, 1.0, 0.02, False, 95)]
    items, refs = [], []
    for p in probs:
        go = make_grad_out(p)
        B = make_weight(p)
        items.append((to_device_go(go, p.go_dtype), nb().quantize(torch.from_numpy(B).cuda()), None))
        data_o, scales_o = oracle.quantize(B)
        go16 = oracle.round_operand(go, p.go_dtype)
        bt = oracle.dequantize_f16(scales_o, data_o, p.K, p.N)
        rows = sample_rows(p.M, 8, p.seed)
        refs.append((rows,) + oracle.backward_a_rows(go16, bt, rows))
    # One problem given in f16 (read in place: no pass, no counters).
    pf = Problem(700, 320, 512, F32, 1.0, 0.02, False, 96)
    items.append((torch.from_numpy(oracle.f32_to_f16(make_grad_out(pf)).view(np.int16)).cuda()
                  .view(torch.float16), nb().quantize(torch.from_numpy(make_weight(pf)).cuda()),
                  None))
    full = nb().batched_ws_workspace(items)
    seq_bytes = _sequential_ws_bytes(items)
    assert full.numel() > seq_bytes
    streamed = nb().backward_a_batched_ws(items, full)
    sequential = nb().backward_a_batched_ws(items, full[:seq_bytes])
    again = nb().backward_a_batched_ws(items, full)
    nb().check_error()
    for i, (a, b, c) in enumerate(zip(streamed, sequential, again)):
        assert torch.equal(a, b), f"problem {i}: streamed != sequential pass"
        assert torch.equal(a, c), f"problem {i}: not repeatable"
    for p, out, (rows, ref, bound) in zip(probs, streamed, refs):
        assert_close(out.cpu().numpy()[rows], ref, bound, str(p))


def test_grouped_512_token_tiles_with_short_items():
    """Forced 512-token tiles over many short problems (1 to 10 stages of 64),
    so that every pair runs several short items back to back: a whole tile's
    epilogue stages in the two A slots its successor fills third and fourth,
    and the A producer must wait for an older item's hand-back at the start of
    the item after next when the item between has fewer than three stages.
    Every result equals the single call with the same tiles bit for bit and
    the oracle on sampled rows; a second launch repeats the bits."""
    rng = np.random.default_rng(97)
    probs = []
    for i in range(40):
        N = int(rng.choice([64, 128, 192, 256, 640]))
        M = int(rng.choice([512, 1000, 1536]))
        K = int(rng.choice([256, 512]))
        probs.append(Problem(M, N, K, F32, 1.0, 0.02, bool(i % 3 == 0), 3000 + i))
    items, refs = [], []
    for p in probs:
        go = make_grad_out(p)
        B = make_weight(p)
        items.append((to_device_go(go, p.go_dtype), nb().quantize(torch.from_numpy(B).cuda()), None))
        data_o, scales_o = oracle.quantize(B)
        bt = oracle.dequantize_f16(scales_o, data_o, p.K, p.N)
        rows = sample_rows(p.M, 4, p.seed)
        refs.append((rows,) + oracle.backward_a_rows(oracle.round_operand(go, p.go_dtype), bt, rows))
    with nb().tile_rows_forced(512), nb().small_m_max(0):
        ws = nb().batched_ws_workspace(items)
        outs = nb().backward_a_batched_ws(items, ws)
        again = nb().backward_a_batched_ws(items, ws)
        singles = [nb().backward_a_ws(go, w, nb().ws_workspace(p.M, p.N, split=False))
                   for p, (go, w, _) in zip(probs, items)]
    nb().check_error()
    for p, out, out2, single, (rows, ref, bound) in zip(probs, outs, again, singles, refs):
        assert torch.equal(out, out2), p
        assert torch.equal(out, single), p
        assert_close(out.cpu().numpy()[rows], ref, bound, str(p))
