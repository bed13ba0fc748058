"""srwm_forward_host: host buffers in and out, copies overlapping the
recurrence chunk by chunk.  Checked against srwm_forward on the device
(chunk restarts change only fp32 rounding) and against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from self_referential_weight_gb300 import binding, inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def rel(a, b):
    return float(np.abs(np.asarray(a, np.float64) - b).max() / max(np.abs(b).max(), 1e-30))


def device_forward(x, W0, n_lr, smx):
    y, Wf = binding.srwm_forward(torch.from_numpy(x).to(DEV), torch.from_numpy(W0).to(DEV), n_lr, smx)
    torch.cuda.synchronize()
    return y.cpu().numpy(), Wf.cpu().numpy()


def host_forward(x, W0, n_lr, smx, chunk, pinned=True):
    xh, Wh = torch.from_numpy(x), torch.from_numpy(W0)
    if pinned:
        xh, Wh = xh.pin_memory(), Wh.pin_memory()
    y, Wf = binding.srwm_forward_host(xh, Wh, n_lr, smx, chunk_steps=chunk)
    torch.cuda.synchronize()
    assert binding.srwm_last_device_status() == 0
    return y.numpy(), Wf.numpy()


@pytest.mark.parametrize("d", [16, 32, 64])
@pytest.mark.parametrize("n_lr,smx", [(4, False), (1, True)])
@pytest.mark.parametrize("chunk", [1, 32, 50, 0])
def test_host_pipeline_matches(d, n_lr, smx, chunk):
    wl = inputs.Workload("t", 3, 75, 2, d, n_lr, smx, 300 + d + chunk, "normal")
    x, W0 = inputs.make_inputs(wl)
    y, Wf = host_forward(x, W0, n_lr, smx, chunk)
    yd, Wd = device_forward(x, W0, n_lr, smx)
    assert rel(y, yd) <= 1e-5 and rel(Wf, Wd) <= 1e-5
    yo, Wo = oracle.forward(x, W0, n_lr, smx)
    assert rel(y, yo) <= 1e-4 and rel(Wf, Wo) <= 1e-4


def test_host_pipeline_many_streams_and_reuse():
    """The two-warp d = 64 kernel (more than two streams per SM), several
    chunks, twice back to back into one workspace."""
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    wl = inputs.Workload("t", (2 * n_sm) // 8 + 5, 160, 8, 64, 4, False, 320, "normal")
    x, W0 = inputs.make_inputs(wl)
    ws = torch.empty(binding.srwm_forward_host_workspace_bytes(wl.B, wl.T, wl.H, wl.d, 4, 64), dtype=torch.uint8,
                     device=DEV)
    xh, Wh = torch.from_numpy(x).pin_memory(), torch.from_numpy(W0).pin_memory()
    y1, W1 = binding.srwm_forward_host(xh, Wh, 4, chunk_steps=64, workspace=ws)
    y2, W2 = binding.srwm_forward_host(xh, Wh, 4, chunk_steps=64, workspace=ws)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(y1.numpy(), y2.numpy())
    np.testing.assert_array_equal(W1.numpy(), W2.numpy())
    yd, Wd = device_forward(x, W0, 4, False)
    assert rel(y1.numpy(), yd) <= 1e-5 and rel(W1.numpy(), Wd) <= 1e-5


def test_host_pipeline_pageable_and_zero_steps():
    wl = inputs.Workload("t", 2, 40, 3, 32, 4, False, 330, "normal")
    x, W0 = inputs.make_inputs(wl)
    y, Wf = host_forward(x, W0, 4, False, 16, pinned=False)
    yd, Wd = device_forward(x, W0, 4, False)
    assert rel(y, yd) <= 1e-5 and rel(Wf, Wd) <= 1e-5
    x0 = np.zeros((2, 0, 3, 32), np.float32)
    _, W = host_forward(x0, W0, 4, False, 0)
    np.testing.assert_array_equal(W, np.broadcast_to(W0, W.shape))


def test_host_pipeline_rejects_device_memory():
    wl = inputs.Workload("t", 2, 8, 2, 16, 4, False, 340, "normal")
    x, W0 = inputs.make_inputs(wl)
    xd = torch.from_numpy(x).to(DEV)
    ws = torch.empty(binding.srwm_forward_host_workspace_bytes(2, 8, 2, 16, 4, 0), dtype=torch.uint8, device=DEV)
    y = torch.empty(x.shape)
    Wf = torch.empty((2, 2, 52, 16))
    lib = binding._lib()
    rc = lib.srwm_forward_host(xd.data_ptr(), torch.from_numpy(W0).data_ptr(), 2, 8, 2, 16, 4, 0, y.data_ptr(),
                               Wf.data_ptr(), 0, ws.data_ptr(), ws.numel(), None)
    assert rc == 3


@pytest.mark.parametrize("d", [32, 64])
@pytest.mark.parametrize("T", [1, 63, 64, 95, 200, 700, 2056])
def test_host_pipeline_doubling_plan(T, d):
    """The default chunk plan (doubling from 32 steps, an even middle whose
    longest chunk depends on d, halving at the end) over several lengths
    equals srwm_forward within fp32 rounding."""
    wl = inputs.Workload("t", 2, T, 2, d, 1, True, 900 + T + d, "normal")
    x, W0 = inputs.make_inputs(wl)
    y, Wf = host_forward(x, W0, 1, True, 0)
    yd, Wd = binding.srwm_forward(torch.from_numpy(x).to(DEV), torch.from_numpy(W0).to(DEV), 1, True)
    torch.cuda.synchronize()
    yd, Wd = yd.cpu().numpy(), Wd.cpu().numpy()
    assert np.abs(y - yd).max() <= 1e-5 * np.abs(yd).max()
    assert np.abs(Wf - Wd).max() <= 1e-5 * np.abs(Wd).max()


def test_host_pipeline_single_chunk_fewshot():
    """The few-shot workload in full (T = 26: the default plan is one chunk,
    which runs its copies in order on the caller's stream)."""
    wl = inputs.workload("fewshot")
    x, W0 = inputs.make_inputs(wl)
    plan = binding.srwm_debug_chunk_plan(wl.T, wl.d, 0)
    assert plan == [wl.T]
    y, Wf = host_forward(x, W0, wl.n_lr, wl.softmax_input, 0)
    yd, Wd = device_forward(x, W0, wl.n_lr, wl.softmax_input)
    assert rel(y, yd) <= 1e-5 and rel(Wf, Wd) <= 1e-5
    yo, Wo = oracle.forward(x, W0, wl.n_lr, wl.softmax_input)
    assert rel(y, yo) <= 1e-4 and rel(Wf, Wo) <= 1e-4
