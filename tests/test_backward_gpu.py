"""GPU parity of srwm_backward (dL/dx, dL/dW0) against the gradient oracle
(float64 autograd through the step-by-step recurrence), on the same seeded
inputs and cotangents.

Tolerance: max|gpu - oracle| / max|oracle| <= 2e-4 per output.  The gradient
is a sum of T backward steps in fp32, each carrying the forward's own rounding
(<= 1e-4 relative for these lengths) into products with dL/dW; twice the
forward's bound covers both.
"""
import numpy as np
import pytest
import torch

from oracle import srwm_grad
from self_referential_weight_gb300 import binding, inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
TOL = 2e-4


def rel(a, b):
    return float(np.abs(np.asarray(a, np.float64) - b).max() / max(np.abs(b).max(), 1e-30))


def run_bwd(x, W0, n_lr, smx, dy, dWf):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(DEV)
    dx, dW0 = binding.srwm_backward(t(x), t(W0), n_lr, smx, t(dy), None if dWf is None else t(dWf))
    torch.cuda.synchronize()
    return dx.cpu().numpy(), dW0.cpu().numpy()


def check(wl, with_dWf=True):
    x, W0 = inputs.make_inputs(wl)
    dy, dWf = inputs.make_cotangents(wl, with_dWf)
    dx, dW0 = run_bwd(x, W0, wl.n_lr, wl.softmax_input, dy, dWf)
    ox, oW = srwm_grad.grads(x, W0, wl.n_lr, wl.softmax_input, dy, dWf)
    assert rel(dx, ox) <= TOL, rel(dx, ox)
    assert rel(dW0, oW) <= TOL, rel(dW0, oW)


# Segments are 32 steps: T = 75 takes two full segments and a ragged tail.
@pytest.mark.parametrize("d", [16, 32, 64])
@pytest.mark.parametrize("n_lr", [1, 4])
@pytest.mark.parametrize("smx", [False, True])
def test_backward_all_variants(d, n_lr, smx):
    check(inputs.Workload("g", 2, 75, 3, d, n_lr, smx, 300 + d + n_lr + smx, "normal"))


@pytest.mark.parametrize("d", [16, 64])
@pytest.mark.parametrize("T", [1, 2, 31, 32, 33, 64, 65])
def test_backward_step_count_edges(d, T):
    check(inputs.Workload("g", 2, T, 2, d, 4, False, 400 + T, "normal"))


@pytest.mark.parametrize("d", [32, 64])
def test_backward_without_dW_final(d):
    check(inputs.Workload("g", 3, 40, 2, d, 4, True, 500 + d, "normal"), with_dWf=False)


def test_backward_fewshot_episodes():
    """The few-shot structure (one-hot label block, zero query label)."""
    check(inputs.workload("fewshot").with_shape(B=8, H=4))


def test_backward_longer_sequence():
    """Several hundred steps: rounding of the stepped-back state stays within
    one segment, so the error does not grow with T."""
    check(inputs.Workload("g", 1, 400, 2, 64, 4, False, 600, "normal"))


@pytest.mark.parametrize("T", [70, 33])
@pytest.mark.parametrize("d,ctas_per_sm", [(64, 1), (32, 3), (16, 8)])
def test_backward_wrap_schedule(d, ctas_per_sm, T):
    """More streams than the backward kernel's co-resident CTAs (one, three or
    eight per SM for d = 64, 32, 16) selects the wrap-around schedule: streams
    split in two hand W and dL/dW from their later to their earlier part.
    dL/dx equals, bit for bit, two half-batch calls that each fit in one wave
    (W and dL/dW pass through memory unchanged); dL/dW0 agrees within the
    rounding of the sum over b; one head's gradients match the oracle."""
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    H = 4
    slots = ctas_per_sm * n_sm
    B = 2 * ((slots // H) // 2 + 4)   # > slots streams; each half <= slots
    wl = inputs.Workload("g", B, T, H, d, 4, False, 800 + T + d, "normal")
    x, W0 = inputs.make_inputs(wl)
    dy, dWf = inputs.make_cotangents(wl, True)
    dx, dW0 = run_bwd(x, W0, 4, False, dy, dWf)
    hB = B // 2
    dx1, dW01 = run_bwd(x[:hB], W0, 4, False, dy[:hB], dWf[:hB])
    dx2, dW02 = run_bwd(x[hB:], W0, 4, False, dy[hB:], dWf[hB:])
    np.testing.assert_array_equal(dx, np.concatenate([dx1, dx2]))
    assert rel(dW0, dW01.astype(np.float64) + dW02) <= 1e-6
    h = 1
    ox, oW = srwm_grad.grads(x[:, :, h:h + 1], W0[h:h + 1], 4, False, dy[:, :, h:h + 1], dWf[:, h:h + 1])
    assert rel(dx[:, :, h:h + 1], ox) <= TOL and rel(dW0[h:h + 1], oW) <= TOL


@pytest.mark.parametrize("d", [16, 64])
def test_backward_zero_steps(d):
    wl = inputs.Workload("g", 3, 0, 2, d, 4, False, 700, "normal")
    W0 = inputs.make_W0(wl.H, d, 4, wl.seed)
    _, dWf = inputs.make_cotangents(wl.with_shape(T=1))
    x = torch.empty((3, 0, 2, d), device=DEV)
    dx, dW0 = binding.srwm_backward(x, torch.from_numpy(W0).to(DEV), 4, False, x.clone(),
                                    torch.from_numpy(dWf).to(DEV))
    torch.cuda.synchronize()
    np.testing.assert_allclose(dW0.cpu().numpy(), dWf.astype(np.float64).sum(0), rtol=1e-6, atol=1e-6)
    dx, dW0 = binding.srwm_backward(x, torch.from_numpy(W0).to(DEV), 4, False, x.clone())
    torch.cuda.synchronize()
    assert not dW0.cpu().numpy().any()


def test_backward_deterministic():
    wl = inputs.Workload("g", 4, 70, 4, 64, 4, False, 800, "normal")
    x, W0 = inputs.make_inputs(wl)
    dy, dWf = inputs.make_cotangents(wl)
    a = run_bwd(x, W0, 4, False, dy, dWf)
    b = run_bwd(x, W0, 4, False, dy, dWf)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_backward_small_workspace_rejected():
    wl = inputs.Workload("g", 2, 40, 2, 16, 4, False, 900, "normal")
    x, W0 = inputs.make_inputs(wl)
    dy, _ = inputs.make_cotangents(wl, False)
    need = binding.srwm_backward_workspace_bytes(2, 40, 2, 16, 4)
    ws = torch.empty(need - 256, dtype=torch.uint8, device=DEV)
    t = lambda a: torch.from_numpy(a).to(DEV)
    with pytest.raises(binding.SrwmError) as e:
        binding.srwm_backward(t(x), t(W0), 4, False, t(dy), workspace=ws)
    assert e.value.status == 2


@pytest.mark.parametrize("name,h", [("mid", 5), ("rl", 2)])
def test_backward_full_size_sampled_head(name, h):
    """Full-size workload through srwm_backward (the launch a training step
    makes); the oracle recomputes one head over every sequence: that head's
    dL/dx and dL/dW0[h] (heads are independent, so the slice's gradients are
    the full problem's)."""
    wl = inputs.workload(name)
    x, W0 = inputs.make_inputs(wl)
    dy, _ = inputs.make_cotangents(wl, False)
    dx, dW0 = run_bwd(x, W0, wl.n_lr, wl.softmax_input, dy, None)
    xs = np.ascontiguousarray(x[:, :, h:h + 1])
    ox, oW = srwm_grad.grads(xs, W0[h:h + 1], wl.n_lr, wl.softmax_input, np.ascontiguousarray(dy[:, :, h:h + 1]))
    assert rel(dx[:, :, h:h + 1], ox) <= TOL, rel(dx[:, :, h:h + 1], ox)
    assert rel(dW0[h:h + 1], oW) <= TOL, rel(dW0[h:h + 1], oW)


def test_backward_long_one_stream():
    """The long workload (T = 8192, where recovering W_{t-1} by subtracting
    each recorded update accumulates the most rounding) at full size through
    srwm_backward, with dy zero on every stream but one.  The other streams'
    gradients are then exactly zero, and dL/dW0[h] is that one stream's
    contribution, which the oracle computes on the (b, h) slice alone.  The
    bar is twice the forward's bound at this length (1e-3)."""
    wl = inputs.workload("long")
    b, h = 11, 6
    x, W0 = inputs.make_inputs(wl)
    dy, _ = inputs.make_cotangents(wl, False)
    mask = np.zeros_like(dy)
    mask[b, :, h] = 1.0
    dy = dy * mask
    dx, dW0 = run_bwd(x, W0, wl.n_lr, wl.softmax_input, dy, None)
    ox, oW = srwm_grad.grads(np.ascontiguousarray(x[b:b + 1, :, h:h + 1]), W0[h:h + 1], wl.n_lr, wl.softmax_input,
                             np.ascontiguousarray(dy[b:b + 1, :, h:h + 1]))
    ex, ew = rel(dx[b:b + 1, :, h:h + 1], ox), rel(dW0[h:h + 1], oW)
    print(f"long backward, stream ({b}, {h}): dx rel {ex:.2e}, dW0 rel {ew:.2e}")
    assert ex <= 2e-3 and ew <= 2e-3, (ex, ew)
    others = np.ones(dx.shape, bool)
    others[b, :, h] = False
    assert not dx[others].any()
    assert not np.delete(dW0, h, axis=0).any()
