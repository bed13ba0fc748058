"""Pins of the gradient oracle (oracle/srwm_grad.py).

The gradient oracle differentiates a second, PyTorch float64 transcription
of the forward recurrence with autograd.  Pinned here:
  * its forward equals the C oracle's (two independent transcriptions);
  * gradients equal central finite differences of the C oracle's loss;
  * T = 1 closed form: y_0 = W0^y x~_0 comes from the pre-update matrix, so
    dL/dW0 = dy (outer) x~_0 on the y rows and zero elsewhere, dL/dx~ = W0^y' dy;
  * one learning rate vs four with copied beta rows: the copies' gradients
    add up to the single row's gradient, all other gradients are equal.
Sources: "Metalearning Continual Learning Algorithms", section 2.3,
Eqs. (1)-(5); review "SRWM:让权重矩阵学习修改自身", section 2.2 (time order).
"""
import numpy as np
import pytest
import torch
from scipy.special import softmax as sp_softmax

import oracle
from oracle import srwm_grad


def _rng(s):
    return np.random.default_rng(s)


def _case(seed, B, T, H, d, n_lr, scale=1.0):
    r = _rng(seed)
    x = (scale * r.standard_normal((B, T, H, d))).astype(np.float32)
    W0 = (r.standard_normal((H, 3 * d + n_lr, d)) / np.sqrt(d)).astype(np.float32)
    dy = r.standard_normal((B, T, H, d))
    dWf = r.standard_normal((B, H, 3 * d + n_lr, d))
    return x, W0, dy, dWf


@pytest.mark.parametrize("n_lr,smx", [(1, False), (4, False), (1, True), (4, True)])
def test_torch_forward_matches_c_oracle(n_lr, smx):
    x, W0, _, _ = _case(1, 2, 12, 3, 5, n_lr)
    y, Wf = srwm_grad.forward_torch(torch.tensor(x, dtype=torch.float64),
                                    torch.tensor(W0, dtype=torch.float64), n_lr, smx)
    yo, Wo = oracle.forward(x, W0, n_lr, smx)
    assert np.abs(y.numpy() - yo).max() <= 1e-12 * np.abs(yo).max()
    assert np.abs(Wf.numpy() - Wo).max() <= 1e-12 * np.abs(Wo).max()


def _loss_c(x, W0, n_lr, smx, dy, dWf):
    y, Wf = oracle.forward(x.astype(np.float32), W0.astype(np.float32), n_lr, smx)
    return float((y * dy).sum() + (Wf * dWf).sum())


@pytest.mark.parametrize("n_lr,smx", [(1, False), (4, True)])
def test_gradients_match_finite_differences(n_lr, smx):
    """Directional derivatives of the C oracle's loss.  The C oracle takes fp32
    inputs, so the probe uses directions and steps that are exact in fp32:
    dyadic base values, a step of 2^-10 along one coordinate at a time."""
    d, T = 3, 5
    x, W0, dy, dWf = _case(2, 1, T, 1, d, n_lr, scale=0.5)
    x = (np.round(x * 64) / 64).astype(np.float32)
    W0 = (np.round(W0 * 64) / 64).astype(np.float32)
    dx, dW0 = srwm_grad.grads(x, W0, n_lr, smx, dy, dWf)
    h = 2.0 ** -10
    r = _rng(3)
    for _ in range(6):
        idx = tuple(int(r.integers(n)) for n in W0.shape)
        Wp, Wm = W0.copy(), W0.copy()
        Wp[idx] += h
        Wm[idx] -= h
        fd = (_loss_c(x, Wp, n_lr, smx, dy, dWf) - _loss_c(x, Wm, n_lr, smx, dy, dWf)) / (2 * h)
        assert abs(fd - dW0[idx]) <= 1e-5 * (1 + abs(dW0[idx])), (idx, fd, dW0[idx])
    for _ in range(6):
        idx = tuple(int(r.integers(n)) for n in x.shape)
        xp, xm = x.copy(), x.copy()
        xp[idx] += h
        xm[idx] -= h
        fd = (_loss_c(xp, W0, n_lr, smx, dy, dWf) - _loss_c(xm, W0, n_lr, smx, dy, dWf)) / (2 * h)
        assert abs(fd - dx[idx]) <= 1e-5 * (1 + abs(dx[idx])), (idx, fd, dx[idx])


@pytest.mark.parametrize("smx", [False, True])
def test_single_step_closed_form(smx):
    d = 6
    x, W0, dy, _ = _case(4, 1, 1, 2, d, 4)
    dx, dW0 = srwm_grad.grads(x, W0, 4, smx, dy)
    xs = x.astype(np.float64)
    if smx:
        xs = sp_softmax(xs, axis=-1)
    want = np.zeros_like(dW0)
    for h in range(2):
        want[h, :d] = np.outer(dy[0, 0, h], xs[0, 0, h])
    np.testing.assert_allclose(dW0, want, atol=1e-12)
    dxs = np.einsum("hod,ho->hd", W0[:, :d].astype(np.float64), dy[0, 0])
    if smx:   # softmax backward: s * (g - <s, g>)
        s = xs[0, 0]
        dxs = s * (dxs - (s * dxs).sum(-1, keepdims=True))
    np.testing.assert_allclose(dx[0, 0], dxs, atol=1e-12)


def test_one_rate_equals_four_rates_gradients():
    d, T = 4, 9
    x, W1, dy, _ = _case(5, 2, T, 2, d, 1)
    W4 = np.concatenate([W1[:, :3 * d], np.repeat(W1[:, 3 * d:], 4, axis=1)], axis=1)
    dx1, dW1 = srwm_grad.grads(x, W1, 1, False, dy)
    dx4, dW4 = srwm_grad.grads(x, W4, 4, False, dy)
    np.testing.assert_allclose(dx4, dx1, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dW4[:, :3 * d], dW1[:, :3 * d], rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dW4[:, 3 * d:].sum(1), dW1[:, 3 * d], rtol=1e-10, atol=1e-12)
