"""Degenerate cases of the recurrence on the GPU, checked through properties
that hold at any size ("Metalearning Continual Learning Algorithms",
section 2.3, Eqs. (1)-(5)):
  * k rows equal to q rows: phi(k) = phi(q) bit for bit, so u = 0 and W never
    changes: W_final = W0 exactly and y_t = W0^y x~_t (a plain matmul);
  * with the input softmax, beta rows of -60: every gate sigma(-60) ~ 9e-27,
    so W_final = W0 bit for bit and again y_t = W0^y x~_t;
  * saturating inputs (x scaled by 5 and 25): near one-hot softmaxes, against
    the oracle within a few times the problem's own fp32 floor;
  * uniform softmaxes (all k rows of W0 equal, and constant x on some steps
    with the input softmax): the kernels' fixed-point sums of exponentials
    reach their largest value, d terms of exactly 1.
"""
import numpy as np
import pytest
import torch

import oracle
from self_referential_weight_gb300 import binding, inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def rel(a, b):
    return float(np.abs(np.asarray(a, np.float64) - b).max() / max(np.abs(b).max(), 1e-30))


def run(x, W0, n_lr, smx):
    y, Wf = binding.srwm_forward(torch.from_numpy(x).to(DEV), torch.from_numpy(W0).to(DEV), n_lr, smx)
    torch.cuda.synchronize()
    assert binding.srwm_last_device_status() == 0
    return y.cpu().numpy(), Wf.cpu().numpy()


def y_rows_matmul(x, W0, smx):
    d = x.shape[-1]
    xt = x.astype(np.float64)
    if smx:
        e = np.exp(xt - xt.max(-1, keepdims=True))
        xt = e / e.sum(-1, keepdims=True)
    return np.einsum("hrc,bthc->bthr", W0[:, :d].astype(np.float64), xt)


@pytest.mark.parametrize("name", ["mid", "rl", "fewshot"])
def test_equal_key_and_query_rows_freeze_W(name):
    wl = inputs.workload(name)
    x, W0 = inputs.make_inputs(wl)
    d = wl.d
    W0 = W0.copy()
    W0[:, 2 * d:3 * d] = W0[:, d:2 * d]
    y, Wf = run(x, W0, wl.n_lr, wl.softmax_input)
    np.testing.assert_array_equal(Wf, np.broadcast_to(W0, Wf.shape))
    assert rel(y, y_rows_matmul(x, W0, wl.softmax_input)) <= 1e-5


@pytest.mark.parametrize("d", [16, 32, 64])
@pytest.mark.parametrize("n_lr", [1, 4])
def test_closed_gates_keep_W0(d, n_lr):
    """With the input softmax x~ sums to 1, so beta rows of -60 give beta = -60
    at every step: the gates sigma(-60) ~ 9e-27 leave every update below half
    an ulp of W, so W_final = W0 bit for bit and y_t = W0^y x~_t."""
    wl = inputs.Workload("t", 4, 70, 3, d, n_lr, True, 60 + d + n_lr, "normal")
    x, W0 = inputs.make_inputs(wl)
    W0 = W0.copy()
    W0[:, 3 * d:, :] = -60.0
    y, Wf = run(x, W0, n_lr, True)
    np.testing.assert_array_equal(Wf, np.broadcast_to(W0, Wf.shape))
    assert rel(y, y_rows_matmul(x, W0, True)) <= 1e-5


@pytest.mark.parametrize("d,n_lr,smx", [(16, 4, False), (16, 1, True), (32, 1, False), (64, 4, False), (64, 1, True)])
@pytest.mark.parametrize("scale", [5.0, 25.0])
def test_saturating_inputs(d, n_lr, smx, scale):
    """Inputs scaled up drive the softmaxes towards one-hot, where the
    recurrence amplifies rounding: at scale 25 the oracle's own float32 run
    differs from its float64 run by up to 1e-3 - 7e-2.  The bound is therefore
    a few times that measured fp32 floor (and never tighter than 1e-4)."""
    wl = inputs.Workload("t", 3, 60, 2, d, n_lr, smx, 80 + d, "normal")
    x, W0 = inputs.make_inputs(wl)
    x = (x * scale).astype(np.float32)
    y, Wf = run(x, W0, n_lr, smx)
    yo, Wo = oracle.forward(x, W0, n_lr, smx)
    y32, W32 = oracle.forward(x, W0, n_lr, smx, precision="f32")
    assert rel(y, yo) <= max(1e-4, 4 * rel(y32, yo))
    assert rel(Wf, Wo) <= max(1e-4, 4 * rel(W32, Wo))


@pytest.mark.parametrize("d", [16, 32, 64])
@pytest.mark.parametrize("smx", [False, True])
def test_uniform_softmaxes(d, smx):
    """All k rows of W0 equal: equal rows get equal updates (same block, same
    gate, same a), so k_t has d equal entries at every step and phi(k_t) is
    exactly uniform; every exponential is 1 and the fixed-point sums reach
    their largest value (at d = 16, 16 * 2^27 = 2^31).  With the input softmax,
    every seventh step's x is constant, so x~ is uniform there too.  Against
    the oracle at the parity bar."""
    wl = inputs.Workload("t", 3, 70, 2, d, 4, smx, 90 + d, "normal")
    x, W0 = inputs.make_inputs(wl)
    W0, x = W0.copy(), x.copy()
    W0[:, d:2 * d] = W0[:, d:d + 1]
    if smx:
        x[:, ::7] = 0.5
    y, Wf = run(x, W0, 4, smx)
    assert np.all(Wf[:, :, d:2 * d] == Wf[:, :, d:d + 1])   # the k rows stay equal
    yo, Wo = oracle.forward(x, W0, 4, smx)
    assert rel(y, yo) <= 1e-4
    assert rel(Wf, Wo) <= 1e-4
