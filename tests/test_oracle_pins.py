"""Pins of the CPU oracle against what the pages and the mathematics fix.

None of these tests re-types the oracle's own formulas: each checks it against
an independent fact -- a published construction (the NF4 quantiles), a library
routine (numpy's IEEE f16 conversion, torch's bf16 widening, numpy float32
arithmetic, torch.matmul in fp64, exact rational arithmetic), an invariant or a
hand-worked layout example from page "aprender-gpu 0.32.0 --
src/kernels/backward/nf4_tensor_core.rs" (build_ptx, "PHASE 2").
"""
from __future__ import annotations

import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from workloads import BF16, F32, Problem, make_grad_out, make_weight

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- codebook
def test_codebook_invariants():
    L = oracle.codebook()
    assert L.dtype == np.float32 and L.shape == (16,)
    assert np.all(np.diff(L) > 0), "strictly increasing"
    assert L[0] == -1.0 and L[7] == 0.0 and L[15] == 1.0
    assert int((L < 0).sum()) == 7 and int((L > 0).sum()) == 8


def test_codebook_matches_normal_quantile_construction():
    """QLoRA's NF4: quantiles of N(0,1) at evenly spaced probabilities from
    p_max = 1 - (1/32 + 1/30)/2 down to 1/2 -- 8 on the positive side, 7 on the
    negative side -- plus an exact zero, each side divided by its largest
    quantile so the ends are exactly +-1."""
    from scipy.stats import norm

    p_max = 1.0 - 0.5 * (1.0 / 32.0 + 1.0 / 30.0)
    pos = norm.ppf(np.linspace(p_max, 0.5, 9)[:-1])
    neg = -norm.ppf(np.linspace(p_max, 0.5, 8)[:-1])
    vals = np.sort(np.concatenate([pos, [0.0], neg]))
    vals = vals / np.max(np.abs(vals))
    L = oracle.codebook().astype(np.float64)
    # The published table was computed in single precision: agree to f32 level.
    np.testing.assert_allclose(L, vals, rtol=0, atol=2e-6)


# ---------------------------------------------------------------- f16 / bf16
def _edge_f32():
    f = np.float32
    vals = [0.0, -0.0, 1.0, -1.0, 65504.0, 65519.99, 65520.0, -65520.0, 1e30, -1e30,
            np.inf, -np.inf, 6.103515625e-05, 6.1e-05, 5.960464477539063e-08,
            2.9802322387695312e-08, 2.98023259e-08, 2.9802321e-08, 1e-8, 1e-40, -1e-45,
            3.0517578125e-05, 1.0009765625, 1.00048828125, 1.000488340854645,
            1.0014648437, 2047.5, 2048.5, 0.333333343]
    return np.array(vals, dtype=f)


def test_f32_to_f16_matches_numpy_ieee():
    rng = np.random.default_rng(0)
    # Random bit patterns over the whole finite f32 range, plus dense coverage
    # of the f16 normal/subnormal range and exact halfway cases.
    bits = rng.integers(0, 2**32, size=200_000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    h = rng.integers(0, 0x7C00, size=50_000).astype(np.uint16)
    mids = (h.view(np.float16).astype(np.float32).view(np.uint32) + np.uint32(1 << 12))
    mids = mids.view(np.float32)  # f16 value + half an f16 ulp (for normals)
    near = (rng.standard_normal(100_000) * rng.choice([1e-6, 1e-3, 1.0, 1e3, 3e4],
                                                      100_000)).astype(np.float32)
    allx = np.concatenate([x, mids, -mids, near, _edge_f32()])
    got = oracle.f32_to_f16(allx)
    with np.errstate(over="ignore"):
        want = allx.astype(np.float16).view(np.uint16)
    np.testing.assert_array_equal(got, want)


def test_f32_to_f16_nan_stays_nan():
    got = oracle.f32_to_f16(np.array([np.nan, -np.nan], dtype=np.float32))
    assert np.all(np.isnan(got.view(np.float16)))


def test_f16_to_f64_matches_numpy():
    h = np.arange(0, 65536, 7, dtype=np.uint32).astype(np.uint16)
    h = h[~np.isnan(h.view(np.float16))]
    got = oracle.f16_to_f64(h)
    want = h.view(np.float16).astype(np.float64)
    np.testing.assert_array_equal(got, want)


def test_bf16_to_f32_matches_torch():
    rng = np.random.default_rng(1)
    b = rng.integers(0, 65536, size=4000).astype(np.uint16)
    want = torch.from_numpy(b.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    got = oracle.bf16_to_f32(b)
    finite = np.isfinite(want)
    np.testing.assert_array_equal(got[finite].view(np.uint32), want[finite].view(np.uint32))


# ---------------------------------------------------------------- quantiser
def _numpy_nearest_codes(B: np.ndarray):
    """Independent float32 brute force: per (block, column) absmax, then the
    codebook entry with the smallest |y - L[c]| (first, i.e. lowest, on ties)."""
    L = oracle.codebook()
    K, N = B.shape
    codes = np.zeros((K, N), dtype=np.int64)
    scales = np.zeros((N, K // 64), dtype=np.float32)
    for b in range(K // 64):
        blk = B[64 * b:64 * (b + 1)]
        s = np.max(np.abs(blk), axis=0).astype(np.float32)
        scales[:, b] = s
        with np.errstate(invalid="ignore", divide="ignore"):
            y = (blk / s[None, :]).astype(np.float32)
        d = np.abs(y[..., None] - L[None, None, :]).astype(np.float32)
        c = np.argmin(d, axis=-1)
        c[:, s == 0] = 7
        codes[64 * b:64 * (b + 1)] = c
    return codes, scales


def _unpack(data: np.ndarray, K: int) -> np.ndarray:
    """codes[k, n] from packed data [N, K/2], read by the page's layout rule."""
    lo = data & 0xF
    hi = data >> 4
    codes_nk = np.stack([lo, hi], axis=-1).reshape(data.shape[0], K)
    return codes_nk.T.astype(np.int64)


def test_quantize_matches_float32_bruteforce():
    rng = np.random.default_rng(2)
    B = (rng.standard_normal((256, 48)) * 0.02).astype(np.float32)
    B[5, 3] = 0.5  # an outlier in one block
    data, scales = oracle.quantize(B)
    want_codes, want_scales = _numpy_nearest_codes(B)
    np.testing.assert_array_equal(scales, want_scales)
    np.testing.assert_array_equal(_unpack(data, 256), want_codes)


def test_quantize_golden_layout():
    with open(os.path.join(GOLDEN, "nf4_layout_k128_n2.json")) as f:
        g = json.load(f)
    K, N = g["K"], g["N"]
    L = oracle.codebook()
    sc = np.array(g["scales"], dtype=np.float32)
    B = np.zeros((K, N), dtype=np.float32)
    for k in range(K):
        for n in range(N):
            B[k, n] = sc[n, k // 64] * L[(k + 5 * n) % 16]
    data, scales = oracle.quantize(B)
    np.testing.assert_array_equal(scales, sc)
    flat = data.reshape(-1)
    for n, idx, byte in g["bytes"]:
        assert flat[idx] == byte, (n, idx)
    for k in range(K):
        for n in range(N):
            assert oracle.code_at(data, K, k, n) == (k + 5 * n) % 16
    bt = oracle.dequantize_f16(scales, data, K, N)
    for k, n, bits in g["dequant_f16_bits"]:
        assert bt[n, k] == bits, (k, n)


def test_quantize_absmax_element_maps_to_an_end_code():
    rng = np.random.default_rng(3)
    B = (rng.standard_normal((128, 40)) * 0.02).astype(np.float32)
    data, scales = oracle.quantize(B)
    codes = _unpack(data, 128)
    for b in range(2):
        blk = B[64 * b:64 * (b + 1)]
        arg = np.argmax(np.abs(blk), axis=0)
        for n in range(40):
            v = blk[arg[n], n]
            c = codes[64 * b + arg[n], n]
            assert c == (15 if v > 0 else 0)
            assert scales[n, b] == abs(v)


def test_quantize_roundtrip_within_half_gap():
    rng = np.random.default_rng(4)
    B = (rng.standard_normal((192, 64)) * 0.02).astype(np.float32)
    data, scales = oracle.quantize(B)
    L = oracle.codebook().astype(np.float64)
    codes = _unpack(data, 192)
    gaps = np.diff(L)
    for k in range(192):
        for n in range(0, 64, 7):
            s = float(scales[n, k // 64])
            c = codes[k, n]
            err = abs(float(B[k, n]) - s * L[c])
            left = gaps[c - 1] if c > 0 else 0.0
            right = gaps[c] if c < 15 else 0.0
            assert err <= 0.5 * max(left, right) * s * (1 + 1e-6) + 1e-12


def test_quantize_zero_block_and_exact_codes():
    L = oracle.codebook()
    K, N = 128, 16
    B = np.zeros((K, N), dtype=np.float32)
    # Block 1 of every column: value L[c] * s for c = k % 16 -> codes come back exactly.
    s = np.float32(0.125)
    for k in range(64, 128):
        B[k, :] = L[k % 16] * s
    data, scales = oracle.quantize(B)
    codes = _unpack(data, K)
    assert np.all(scales[:, 0] == 0) and np.all(codes[:64] == 7)
    assert np.all(scales[:, 1] == s)
    assert np.all(codes[64:] == (np.arange(64, 128) % 16)[:, None])


# ---------------------------------------------------------------- dequant
def test_dequant_matches_numpy_float32_then_f16():
    rng = np.random.default_rng(5)
    B = (rng.standard_normal((128, 24)) * 0.02).astype(np.float32)
    B[::17, 3] *= 20
    data, scales = oracle.quantize(B)
    bt = oracle.dequantize_f16(scales, data, 128, 24)
    L = oracle.codebook()
    codes = _unpack(data, 128)
    want = np.empty((24, 128), dtype=np.uint16)
    for n in range(24):
        for k in range(128):
            w = np.float32(scales[n, k // 64]) * L[codes[k, n]]  # numpy f32 multiply
            want[n, k] = np.array([w], dtype=np.float32).astype(np.float16).view(np.uint16)[0]
    np.testing.assert_array_equal(bt, want)


# ---------------------------------------------------------------- GEMM
def _small_case(M, N, K, dtype=F32, seed=7):
    p = Problem(M, N, K, dtype, 1.0, 0.02, False, seed)
    go = make_grad_out(p)
    data, scales = oracle.quantize(make_weight(p))
    return p, go, data, scales


def test_gemm_bruteforce_exact_16x16x64():
    """Exact rational sum of the f16 operand products vs the fp64 oracle."""
    p, go, data, scales = _small_case(16, 16, 64)
    ref, bound = oracle.backward_a(go, F32, scales, data, 64)
    go16 = oracle.round_operand(go, F32).view(np.float16).astype(np.float64)
    bt = oracle.dequantize_f16(scales, data, 64, 16).view(np.float16).astype(np.float64)
    for m in range(16):
        for k in range(64):
            exact = sum(Fraction(go16[m, n]) * Fraction(bt[n, k]) for n in range(16))
            assert abs(ref[m, k] - float(exact)) <= 1e-15 * bound[m, k] + 1e-300
            ab = sum(abs(Fraction(go16[m, n]) * Fraction(bt[n, k])) for n in range(16))
            assert bound[m, k] == pytest.approx(float(ab), rel=1e-15)


def test_gemm_matches_torch_fp64_matmul():
    for dtype in (F32, BF16):
        p, go, data, scales = _small_case(40, 96, 192, dtype, seed=11)
        ref, _ = oracle.backward_a(go, dtype, scales, data, 192, want_bound=False)
        go16 = oracle.round_operand(go, dtype).view(np.float16).astype(np.float64)
        bt = oracle.dequantize_f16(scales, data, 192, 96).view(np.float16).astype(np.float64)
        want = torch.from_numpy(go16) @ torch.from_numpy(bt)  # [M,N] @ [N,K]
        np.testing.assert_allclose(ref, want.numpy(), rtol=1e-12, atol=1e-300)


def test_gemm_bf16_operand_is_widened_then_rounded():
    p, go, data, scales = _small_case(8, 64, 64, BF16, seed=3)
    widened = torch.from_numpy(go.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    np.testing.assert_array_equal(oracle.round_operand(go, BF16),
                                  widened.astype(np.float16).view(np.uint16))


def test_gemm_one_hot_rows_recover_dequantised_columns():
    K, N = 192, 80
    _, _, data, scales = _small_case(1, N, K, seed=13)
    bt = oracle.dequantize_f16(scales, data, K, N).view(np.float16).astype(np.float64)
    ns = [0, 1, 15, 16, 63, 64, 79]
    go = np.zeros((len(ns), N), dtype=np.float32)
    for i, n in enumerate(ns):
        go[i, n] = 1.0
    ref, _ = oracle.backward_a(go, F32, scales, data, K)
    for i, n in enumerate(ns):
        np.testing.assert_array_equal(ref[i], bt[n])


def test_gemm_linearity_and_zero():
    p, go, data, scales = _small_case(12, 64, 128, seed=17)
    go = np.round(go * 8) / 8  # exactly representable in f16, so rounding is the identity
    ref1, _ = oracle.backward_a(go, F32, scales, data, 128)
    ref2, _ = oracle.backward_a((2 * go).astype(np.float32), F32, scales, data, 128)
    np.testing.assert_array_equal(ref2, 2 * ref1)
    refz, _ = oracle.backward_a(np.zeros_like(go), F32, scales, data, 128)
    assert np.all(refz == 0)
    # Additivity over a split of the shared dimension N.
    go_a = go.copy(); go_a[:, 32:] = 0
    go_b = go.copy(); go_b[:, :32] = 0
    ra, _ = oracle.backward_a(go_a, F32, scales, data, 128)
    rb, _ = oracle.backward_a(go_b, F32, scales, data, 128)
    np.testing.assert_allclose(ra + rb, ref1, rtol=1e-13, atol=1e-300)


def test_rows_entry_matches_full():
    p, go, data, scales = _small_case(33, 64, 128, seed=19)
    ref, bound = oracle.backward_a(go, F32, scales, data, 128)
    go16 = oracle.round_operand(go, F32)
    bt = oracle.dequantize_f16(scales, data, 128, 64)
    rows = [0, 5, 32]
    r, b = oracle.backward_a_rows(go16, bt, rows)
    np.testing.assert_array_equal(r, ref[rows])
    np.testing.assert_array_equal(b, bound[rows])


def test_oracle_rejects_bad_arguments():
    with pytest.raises(ValueError):
        oracle.quantize(np.zeros((100, 4), dtype=np.float32))  # K % 64 != 0
    go16 = np.zeros((4, 8), dtype=np.uint16)
    bt = np.zeros((8, 64), dtype=np.uint16)
    with pytest.raises(ValueError):
        oracle.backward_a_rows(go16, bt, [4])  # row out of range


# ---------------------------------------------------------------- forward product
def _fwd_case(M, N, K, dtype=F32, seed=23):
    """A [M, K] and an NF4 weight B [K, N]: the forward product's inputs (the
    backward's generators with the roles of N and K swapped for A)."""
    p = Problem(M, K, N, dtype, 1.0, 0.02, False, seed)
    a = make_grad_out(p)  # [M, K]
    w = make_weight(Problem(M, N, K, dtype, 1.0, 0.02, False, seed + 1))  # [K, N]
    data, scales = oracle.quantize(w)
    return a, data, scales


def test_forward_bruteforce_exact_8x16x64():
    """Exact rational sum over k of the f16 operand products vs the fp64 oracle."""
    M, N, K = 8, 16, 64
    a, data, scales = _fwd_case(M, N, K)
    ref, bound = oracle.forward(a, F32, scales, data, N)
    a16 = oracle.round_operand(a, F32).view(np.float16).astype(np.float64)
    bt = oracle.dequantize_f16(scales, data, K, N).view(np.float16).astype(np.float64)
    for m in range(M):
        for n in range(N):
            prods = [Fraction(a16[m, k]) * Fraction(bt[n, k]) for k in range(K)]
            assert abs(ref[m, n] - float(sum(prods))) <= 1e-15 * bound[m, n] + 1e-300
            assert bound[m, n] == pytest.approx(float(sum(abs(x) for x in prods)), rel=1e-15)


def test_forward_matches_torch_fp64_matmul():
    for dtype in (F32, BF16):
        M, N, K = 24, 80, 256
        a, data, scales = _fwd_case(M, N, K, dtype, seed=29)
        ref, _ = oracle.forward(a, dtype, scales, data, N, want_bound=False)
        a16 = oracle.round_operand(a, dtype).view(np.float16).astype(np.float64)
        deq = oracle.dequantize_f16(scales, data, K, N).view(np.float16).astype(np.float64).T
        want = torch.from_numpy(a16) @ torch.from_numpy(np.ascontiguousarray(deq))  # [M,K]@[K,N]
        np.testing.assert_allclose(ref, want.numpy(), rtol=1e-12, atol=1e-300)


def test_forward_one_hot_rows_recover_dequantised_rows():
    """A row e_k picks row k of deq(B) [K x N]: C[m, n] = deq(B)[k, n] exactly,
    across block (64) and tile boundaries and odd and even k."""
    M, N, K = 1, 96, 320
    _, data, scales = _fwd_case(M, N, K, seed=31)
    bt = oracle.dequantize_f16(scales, data, K, N).view(np.float16).astype(np.float64)
    ks = [0, 1, 62, 63, 64, 65, 127, 128, 255, 256, 319]
    a = np.zeros((len(ks), K), dtype=np.float32)
    for i, k in enumerate(ks):
        a[i, k] = 1.0
    ref, _ = oracle.forward(a, F32, scales, data, N)
    for i, k in enumerate(ks):
        np.testing.assert_array_equal(ref[i], bt[:, k])


def test_forward_rows_entry_matches_full():
    a, data, scales = _fwd_case(17, 32, 128, seed=37)
    ref, bound = oracle.forward(a, F32, scales, data, 32)
    r, b = oracle.forward_rows(oracle.round_operand(a, F32),
                               oracle.dequantize_f16(scales, data, 128, 32), [0, 9, 16])
    np.testing.assert_array_equal(r, ref[[0, 9, 16]])
    np.testing.assert_array_equal(b, bound[[0, 9, 16]])


# ---------------------------------------------------------------- fused sibling projections
# grad_x = sum_p f16(go_p) @ deq(B_p)^T over projections that share the layer
# input (q/k/v, gate/up): page "aprender-gpu 0.32.0 -- src/kernels/backward/
# nf4_tensor_core.rs", struct doc comment (7 backward projections per layer)
# and the Qwen-dimension test (q/k/v and gate/up share the input width).
def _fused_case(M, Ns, K, seed):
    go16s, bts = [], []
    for j, N in enumerate(Ns):
        p, go, data, scales = _small_case(M, N, K, seed=seed + j)
        go16s.append(oracle.round_operand(go, F32))
        bts.append(oracle.dequantize_f16(scales, data, K, N))
    return go16s, bts


def test_fused_exact_rational_sum():
    M, Ns, K = 5, (16, 8, 24), 64
    go16s, bts = _fused_case(M, Ns, K, 31)
    ref, bound = oracle.backward_a_fused_rows(go16s, bts, np.arange(M))
    g = [x.view(np.float16).astype(np.float64) for x in go16s]
    b = [x.view(np.float16).astype(np.float64) for x in bts]
    for m in range(M):
        for k in range(0, K, 7):
            exact = sum(Fraction(g[p][m, n]) * Fraction(b[p][n, k])
                        for p in range(3) for n in range(Ns[p]))
            assert abs(ref[m, k] - float(exact)) <= 1e-15 * bound[m, k] + 1e-300
            ab = sum(abs(Fraction(g[p][m, n]) * Fraction(b[p][n, k]))
                     for p in range(3) for n in range(Ns[p]))
            assert bound[m, k] == pytest.approx(float(ab), rel=1e-15)


def test_fused_equals_sum_of_separate_products_on_exact_inputs():
    """grad_out values on a coarse grid (multiples of 1/8 up to 4): every product
    and every partial sum is exact in fp64, so the fused sum must equal the sum
    of the separate backward-A products bit for bit."""
    M, Ns, K = 9, (64, 16, 40), 128
    go16s, bts = [], []
    for j, N in enumerate(Ns):
        p, go, data, scales = _small_case(M, N, K, seed=41 + j)
        go = np.clip(np.round(go * 8) / 8, -4, 4).astype(np.float32)
        go16s.append(oracle.round_operand(go, F32))
        bts.append(oracle.dequantize_f16(scales, data, K, N))
    fused, _ = oracle.backward_a_fused_rows(go16s, bts, np.arange(M))
    parts = [oracle.backward_a_rows(g, b, np.arange(M))[0] for g, b in zip(go16s, bts)]
    np.testing.assert_array_equal(fused, parts[0] + parts[1] + parts[2])


def test_fused_one_hot_rows_recover_one_projections_dequantised_columns():
    M, Ns, K = 4, (32, 16, 48), 192
    _, bts = _fused_case(1, Ns, K, 51)
    one = np.float16(1.0).view(np.uint16)
    picks = [(0, 0), (1, 15), (2, 47), (2, 16)]  # (part, n) per row
    go16s = [np.zeros((M, N), dtype=np.uint16) for N in Ns]
    for m, (p, n) in enumerate(picks):
        go16s[p][m, n] = one
    ref, _ = oracle.backward_a_fused_rows(go16s, bts, np.arange(M))
    for m, (p, n) in enumerate(picks):
        np.testing.assert_array_equal(ref[m], bts[p][n].view(np.float16).astype(np.float64))


def test_fused_matches_torch_fp64_matmul_of_the_concatenation():
    M, Ns, K = 20, (96, 32, 32), 256
    go16s, bts = _fused_case(M, Ns, K, 61)
    ref, _ = oracle.backward_a_fused_rows(go16s, bts, np.arange(M), want_bound=False)
    g = np.concatenate([x.view(np.float16).astype(np.float64) for x in go16s], axis=1)
    b = np.concatenate([x.view(np.float16).astype(np.float64) for x in bts], axis=0)
    want = torch.from_numpy(g) @ torch.from_numpy(b)
    np.testing.assert_allclose(ref, want.numpy(), rtol=1e-12, atol=1e-300)


# ---------------------------------------------------------------- dense GemmBackwardB
# grad_B = A^T @ grad_C (page "trueno-gpu 0.4.17 -- src/kernels/backward/mod.rs",
# module list: GEMM gradients for A and B; GemmBackwardBKernel's a_ptr and
# grad_b_ptr parameters), 16-bit operands, fp64 sum over the tokens m.
def _half_case(M, K, N, dtype16, seed):
    g = torch.Generator().manual_seed(seed)
    a = torch.randn(M, K, generator=g) * 0.5
    c = torch.randn(M, N, generator=g) * 0.01
    dt = torch.bfloat16 if dtype16 == oracle.HALF_BF16 else torch.float16
    a, c = a.to(dt), c.to(dt)
    bits = lambda t: t.view(torch.int16).numpy().view(np.uint16)
    return bits(a), bits(c), a.double().numpy(), c.double().numpy()


@pytest.mark.parametrize("dtype16", [oracle.HALF_F16, oracle.HALF_BF16])
def test_gemm_backward_b_exact_rational_sum(dtype16):
    M, K, N = 24, 6, 10
    a, c, af, cf = _half_case(M, K, N, dtype16, 5)
    ref, bound = oracle.gemm_backward_b_rows(a, c, dtype16)
    for k in range(K):
        for n in range(N):
            exact = sum(Fraction(af[m, k]) * Fraction(cf[m, n]) for m in range(M))
            assert abs(ref[k, n] - float(exact)) <= 1e-15 * bound[k, n] + 1e-300
            ab = sum(abs(Fraction(af[m, k]) * Fraction(cf[m, n])) for m in range(M))
            assert bound[k, n] == pytest.approx(float(ab), rel=1e-15)


@pytest.mark.parametrize("dtype16", [oracle.HALF_F16, oracle.HALF_BF16])
def test_gemm_backward_b_matches_torch_fp64(dtype16):
    M, K, N = 300, 40, 72
    a, c, af, cf = _half_case(M, K, N, dtype16, 9)
    ref, _ = oracle.gemm_backward_b_rows(a, c, dtype16, want_bound=False)
    want = torch.from_numpy(af).T @ torch.from_numpy(cf)
    np.testing.assert_allclose(ref, want.numpy(), rtol=1e-12, atol=1e-300)
    # Sampled output rows equal the same rows of the whole result.
    rows = np.array([0, 7, 39], dtype=np.int32)
    sub, _ = oracle.gemm_backward_b_rows(a, c, dtype16, rows=rows)
    np.testing.assert_array_equal(sub, ref[rows])


def test_gemm_backward_b_one_hot_tokens_pick_rows_of_grad_c():
    """A one-hot in column k of token m makes row k of grad_B equal to row m
    of grad_C exactly; a token with A = 0 contributes nothing."""
    M, K, N = 8, 5, 24
    _, c, _, cf = _half_case(M, K, N, oracle.HALF_BF16, 13)
    one = np.uint16(0x3F80)  # bf16 1.0
    a = np.zeros((M, K), dtype=np.uint16)
    picks = {0: 3, 2: 6, 4: 1}  # k -> m
    for k, m in picks.items():
        a[m, k] = one
    ref, _ = oracle.gemm_backward_b_rows(a, c, oracle.HALF_BF16)
    for k in range(K):
        want = cf[picks[k]] if k in picks else np.zeros(N)
        np.testing.assert_array_equal(ref[k], want)
