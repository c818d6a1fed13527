"""Pins of the RMS layer-norm backward oracle (page "trueno-gpu 0.4.17 --
src/kernels/backward/rms_norm.rs", module doc) against what the mathematics
fixes: central finite differences of the stated forward (the page's own
falsifiable prediction) and torch.autograd in fp64."""
from __future__ import annotations

import numpy as np
import torch

from oracle import rms_norm

EPS = 1e-6


def _case(rows=3, H=8, seed=0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((rows, H))
    gamma = rng.standard_normal(H) * 0.5 + 1.0
    g = rng.standard_normal((rows, H))
    return x, gamma, g


def _loss(x, gamma, g):
    y, _ = rms_norm.forward(x, gamma, EPS)
    return float((g * y).sum())


def test_backward_matches_central_finite_differences():
    x, gamma, g = _case()
    _, r = rms_norm.forward(x, gamma, EPS)
    dx, dgamma, _, _ = rms_norm.backward(x, gamma, r, g)
    h = 1e-6
    fd_x = np.zeros_like(x)
    for i in range(x.shape[0]):
        for j in range(x.shape[1]):
            xp, xm = x.copy(), x.copy()
            xp[i, j] += h
            xm[i, j] -= h
            fd_x[i, j] = (_loss(xp, gamma, g) - _loss(xm, gamma, g)) / (2 * h)
    fd_g = np.zeros_like(gamma)
    for j in range(gamma.size):
        gp, gm = gamma.copy(), gamma.copy()
        gp[j] += h
        gm[j] -= h
        fd_g[j] = (_loss(x, gp, g) - _loss(x, gm, g)) / (2 * h)
    np.testing.assert_allclose(dx, fd_x, rtol=1e-6, atol=1e-8)
    np.testing.assert_allclose(dgamma, fd_g, rtol=1e-6, atol=1e-8)


def test_backward_matches_torch_autograd_fp64():
    x, gamma, g = _case(rows=17, H=96, seed=1)
    xt = torch.tensor(x, requires_grad=True)
    gt = torch.tensor(gamma, requires_grad=True)
    r = torch.sqrt((xt * xt).mean(dim=1, keepdim=True) + EPS)
    y = xt * gt / r
    (torch.tensor(g) * y).sum().backward()
    dx, dgamma, _, _ = rms_norm.backward(x, gamma, r.detach().numpy()[:, 0], g)
    np.testing.assert_allclose(dx, xt.grad.numpy(), rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(dgamma, gt.grad.numpy(), rtol=1e-12, atol=1e-14)


def test_page_formula_differs_unless_gamma_is_one():
    """The page's printed dL/dx multiplies the correction term by gamma_i too:
    it matches the gradient only for gamma = 1 (the reading taken here)."""
    x, gamma, g = _case(rows=4, H=16, seed=2)
    _, r = rms_norm.forward(x, gamma, EPS)

    def page(gam):
        rr = r[:, None]
        mean = (x * g * gam[None, :]).mean(axis=1, keepdims=True)
        return gam[None, :] / rr * (g - x / rr ** 2 * mean)

    dx, _, _, _ = rms_norm.backward(x, gamma, r, g)
    assert np.abs(page(gamma) - dx).max() > 1e-3
    ones = np.ones_like(gamma)
    dx1, _, _, _ = rms_norm.backward(x, ones, r, g)
    np.testing.assert_allclose(page(ones), dx1, rtol=1e-12, atol=1e-14)
