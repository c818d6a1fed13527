"""Seeded synthetic workloads for the NF4 backward-A GEMM.

This module only draws numbers: it holds none of the method's arithmetic (no
quantisation, rounding or product).  The tests, the benchmark and the smoke
check feed the same arrays to the CPU oracle and to the CUDA library.

Shapes follow the Qwen2.5-1.5B projections (hidden 1536, KV width 256,
intermediate 8960) that the page "aprender-gpu 0.32.0 --
src/kernels/backward/nf4_tensor_core.rs" uses in its Qwen-dimension test, with
the page's 28 layers x 7 projections for a full training step (struct doc
comment).  Problem (M, N, K): grad_out is [M x N], the NF4 weight B is [K x N],
grad_A is [M x K].

Recipe (the reading of "N(0, s)" is: normal with standard deviation s):
  grad_out ~ N(0, go_std), fp32 or bf16 (bf16 = the fp32 draw rounded by torch).
  B        ~ N(0, b_std), fp32; with ``outliers``, a seeded uniformly random
             0.1% of B's entries are multiplied by 20 before quantisation.
  Seeds: grad_out uses ``seed``, B uses ``seed + 1``; the full step uses
  seed = 1000 * layer + projection index.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

F32 = 0
BF16 = 1
DTYPE_NAMES = {F32: "f32", BF16: "bf16"}


@dataclass(frozen=True)
class Problem:
    M: int
    N: int
    K: int
    go_dtype: int = F32
    go_std: float = 1.0
    b_std: float = 0.02
    outliers: bool = False
    seed: int = 0
    name: str = ""

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def go_bytes(self) -> int:
        return self.M * self.N * (4 if self.go_dtype == F32 else 2)

    @property
    def algorithmic_bytes(self) -> int:
        """grad_out + NF4 codes + fp32 scales + fp32 grad_A (dense B not counted)."""
        return (self.go_bytes + self.K * self.N // 2 + 4 * self.N * (self.K // 64)
                + 4 * self.M * self.K)


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def make_grad_out(p: Problem) -> np.ndarray:
    """fp32 [M, N], or bf16 bits as uint16 [M, N]."""
    g = _gen(p.seed)
    x = torch.randn(p.M, p.N, generator=g, dtype=torch.float32) * p.go_std
    if p.go_dtype == F32:
        return x.numpy()
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def make_weight(p: Problem) -> np.ndarray:
    """Dense fp32 B [K, N] (row-major) before quantisation."""
    g = _gen(p.seed + 1)
    b = torch.randn(p.K, p.N, generator=g, dtype=torch.float32) * p.b_std
    if p.outliers:
        count = max(1, (p.K * p.N) // 1000)
        idx = torch.randperm(p.K * p.N, generator=g)[:count]
        b.view(-1)[idx] *= 20.0
    return b.numpy()


# ---------------------------------------------------------------- configurations
HIDDEN = 1536
KV = 256
INTER = 8960
LAYERS = 28

# (name, N = projection output width, K = projection input width)
QWEN_PROJECTIONS = (
    ("q", HIDDEN, HIDDEN),
    ("k", KV, HIDDEN),
    ("v", KV, HIDDEN),
    ("o", HIDDEN, HIDDEN),
    ("gate", INTER, HIDDEN),
    ("up", INTER, HIDDEN),
    ("down", HIDDEN, INTER),
)


def full_step(M: int = 4096, layers: int = LAYERS) -> list[Problem]:
    out = []
    for layer in range(layers):
        for j, (nm, n, k) in enumerate(QWEN_PROJECTIONS):
            out.append(Problem(M, n, k, F32, 1e-2, 0.02, False, 1000 * layer + j,
                               f"L{layer}.{nm}"))
    return out


# Sibling projections whose input gradients add (they read the same layer
# input): q/k/v and gate/up of one layer, as parts of one fused call; each part
# keeps its own seeded grad_out and weight (layer 0 of the full step).
def fused_parts(names: tuple[str, ...], M: int = 4096, layer: int = 0) -> list[Problem]:
    probs = full_step(M, layers=layer + 1)[7 * layer: 7 * layer + 7]
    return [p for p in probs if p.name.split(".")[1] in names]


FUSED: dict[str, list[Problem]] = {
    "fused_qkv": fused_parts(("q", "k", "v")),
    "fused_gate_up": fused_parts(("gate", "up")),
}

CONFIGS: dict[str, list[Problem]] = {
    "tiny": [Problem(32, 64, 128, F32, 1.0, 0.02, False, 0, "tiny")],
    "q_proj": [Problem(2048, HIDDEN, HIDDEN, F32, 1e-2, 0.02, False, 0, "q_proj")],
    "mlp": [Problem(4096, INTER, HIDDEN, BF16, 1e-2, 0.02, True, 0, "up_proj"),
            Problem(4096, HIDDEN, INTER, BF16, 1e-2, 0.02, True, 2, "down_proj")],
    "full_step": full_step(),
    "large": [Problem(8191, 14336, 4096, F32, 1.0, 0.015, False, 0, "large_a"),
              Problem(8191, 4096, 14336, F32, 1.0, 0.015, False, 2, "large_b"),
              Problem(16, 14336, 4096, F32, 1.0, 0.015, False, 4, "small_m_a"),
              Problem(16, 4096, 14336, F32, 1.0, 0.015, False, 6, "small_m_b")],
}
