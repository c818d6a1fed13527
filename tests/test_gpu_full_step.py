"""The full training step at full size: 28 layers x 7 projections at M = 4096
tokens, fp32 grad_out, as one grouped call (page "aprender-gpu 0.32.0 --
src/kernels/backward/nf4_tensor_core.rs", struct doc comment: 28 layers x 7
backward projections per training step; shapes from the same page's Qwen
dimension test, with Qwen2.5-1.5B's intermediate size 8960).

Every one of the 196 problems is compared with the oracle on sampled rows
(the first and last rows of the 256- and 512-token tiles at the start, a few
seeded random rows and the last row), element by element at the tolerance of
every parity test.  The grouped pre-converted launch and the grouped plain
launch must agree bit for bit, and the seven projections of layers 0, 13 and
27 must equal single unsplit calls bit for bit.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from parity import assert_close, to_device_go
from workloads import CONFIGS, make_grad_out, make_weight

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

WATCH_LAYERS = (0, 13, 27)


@pytest.fixture(scope="module")
def nb():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from backward_gemm_gb300.build import build

    build()
    import backward_gemm_gb300

    backward_gemm_gb300.lib()
    return backward_gemm_gb300


def _rows(M: int, seed: int, extra: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    fixed = {0, 255, 256, 511, 512, M - 1}
    return np.array(sorted({r for r in fixed if r < M} | set(rng.integers(0, M, extra).tolist())),
                    dtype=np.int32)


@pytest.fixture(scope="module")
def full_step(nb):
    """Device inputs of the 196 problems and the oracle's sampled rows.  Each
    problem's host arrays are dropped once its rows are computed."""
    probs = CONFIGS["full_step"]
    items, refs = [], []
    for i, p in enumerate(probs):
        go = make_grad_out(p)
        B = make_weight(p)
        w = nb.quantize(torch.from_numpy(B).cuda())
        items.append((to_device_go(go, p.go_dtype), w))
        data_o, scales_o = oracle.quantize(B)
        bt = oracle.dequantize_f16(scales_o, data_o, p.K, p.N)
        rows = _rows(p.M, p.seed, 8 if (i // 7) in WATCH_LAYERS else 2)
        go16 = oracle.round_operand(go[rows], p.go_dtype)
        ref, bound = oracle.backward_a_rows(go16, bt, np.arange(rows.size, dtype=np.int32))
        refs.append((rows, ref, bound))
    torch.cuda.synchronize()
    return probs, items, refs


def test_full_step_grouped_launches_match_oracle_and_single_calls(nb, full_step):
    probs, items, refs = full_step
    outs_ws = nb.backward_a_batched_ws([(go, w, None) for go, w in items])
    nb.check_error()
    for p, out, (rows, ref, bound) in zip(probs, outs_ws, refs):
        assert_close(out[torch.from_numpy(rows).long().cuda()].cpu().numpy(), ref, bound,
                     f"{p.name} (grouped pre-converted launch)")
    outs_plain = nb.backward_a_batched([(go, w, None) for go, w in items])
    nb.check_error()
    for p, a, b in zip(probs, outs_ws, outs_plain):
        assert torch.equal(a, b), f"{p.name}: grouped launches differ"
    del outs_plain
    for layer in WATCH_LAYERS:
        for j in range(7):
            i = 7 * layer + j
            go, w = items[i]
            p = probs[i]
            single = nb.backward_a_ws(go, w, nb.ws_workspace(p.M, p.N, split=False))
            nb.check_error()
            assert torch.equal(outs_ws[i], single), f"{p.name}: grouped != single call"
