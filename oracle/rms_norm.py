"""RMS layer-norm forward and backward in fp64: the oracle of
``rms_norm_backward``.

TEST INFRASTRUCTURE ONLY (imported by ``tests/``, the smoke check and the
benchmark's CPU legs; the product path never imports it).

Page "trueno-gpu 0.4.17 -- src/kernels/backward/rms_norm.rs", module doc
"Mathematical Specification": per row of H elements the forward is
y_i = x_i * gamma_i / r with r = sqrt(mean(x^2) + eps); the backward gives
dL/dx and dL/dgamma for an upstream gradient g = dL/dy.  Written here from the
chain rule on that forward (which the page's falsifiable prediction, agreement
with finite differences, fixes):

    dL/dx_i = gamma_i g_i / r - x_i mean_j(x_j g_j gamma_j) / r^3
    dL/dgamma_i = sum over rows of g_i x_i / r

The page's printed formula also multiplies the second term by gamma_i and its
kernel adds eps to r^2 again; both are read as defects (the finite-difference
pin in the tests shows the difference).
"""
from __future__ import annotations

import numpy as np


def forward(x: np.ndarray, gamma: np.ndarray, eps: float):
    """y [rows, H] and r [rows] in fp64 (inputs widened exactly)."""
    x = np.asarray(x, dtype=np.float64)
    gamma = np.asarray(gamma, dtype=np.float64)
    r = np.sqrt(np.mean(x * x, axis=1) + eps)
    return x * gamma[None, :] / r[:, None], r


def backward(x: np.ndarray, gamma: np.ndarray, rms: np.ndarray, g: np.ndarray):
    """(dL/dx [rows, H], dL/dgamma [H], bound_x [rows, H], bound_gamma [H]) in
    fp64, from the forward's stored r (rms).  The bounds are the same sums over
    absolute values, for tolerances."""
    x = np.asarray(x, dtype=np.float64)
    g = np.asarray(g, dtype=np.float64)
    gamma = np.asarray(gamma, dtype=np.float64)
    r = np.asarray(rms, dtype=np.float64)[:, None]
    H = x.shape[1]
    xgg = x * g * gamma[None, :]
    mean = xgg.sum(axis=1, keepdims=True) / H
    mean_abs = np.abs(xgg).sum(axis=1, keepdims=True) / H
    dx = gamma[None, :] * g / r - x * mean / r ** 3
    bound_x = np.abs(gamma[None, :] * g) / r + np.abs(x) * mean_abs / r ** 3
    dgamma = (g * x / r).sum(axis=0)
    bound_gamma = np.abs(g * x / r).sum(axis=0)
    return dx, dgamma, bound_x, bound_gamma
