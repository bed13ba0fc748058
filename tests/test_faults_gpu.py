"""Bounded waits: a TMA load that never arrives ends the kernel with a status,
not a hang, and leaves the context usable.

The fault is made on the host: srwm_debug_skip_x_chunk(1) makes the kernels
skip issuing the load of input chunk 1, so the wait for it runs out after the
(shortened) wait limit.  Nothing faults or traps on the GPU.
"""
import numpy as np
import pytest
import torch

import oracle
from self_referential_weight_gb300 import binding, inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture
def short_waits():
    binding.srwm_set_wait_limit_ns(50_000_000)  # 50 ms
    yield
    binding.srwm_debug_skip_x_chunk(-1)
    binding.srwm_set_wait_limit_ns(1_000_000_000)


@pytest.mark.parametrize("d,B,smx", [(16, 2, False), (32, 2, False), (64, 2, False), (64, 110, False),
                                     (64, 110, True)])
def test_missing_chunk_times_out_then_recovers(short_waits, d, B, smx):
    """B = 110 (330 streams at H = 3, more than two per SM on a GB300) runs the
    two-warp d = 64 kernel, whose CTAs agree on a timeout at chunk boundaries,
    with and without the input softmax."""
    wl = inputs.Workload("t", B, 100, 3, d, 4, smx, 40 + d, "normal")
    x, W0 = inputs.make_inputs(wl)
    xd, W0d = torch.from_numpy(x).to(DEV), torch.from_numpy(W0).to(DEV)
    assert binding.srwm_last_device_status() == 0

    binding.srwm_debug_skip_x_chunk(1)
    binding.srwm_forward(xd, W0d, 4, smx)
    assert binding.srwm_last_device_status() == binding.SRWM_ERR_TIMEOUT
    assert binding.srwm_last_device_status() == 0  # reading clears it

    binding.srwm_debug_skip_x_chunk(-1)
    y, Wf = binding.srwm_forward(xd, W0d, 4, smx)
    assert binding.srwm_last_device_status() == 0
    yo, Wo = oracle.forward(x, W0, 4, smx)
    assert np.abs(y.cpu().numpy() - yo).max() / np.abs(yo).max() <= 1e-4
    assert np.abs(Wf.cpu().numpy() - Wo).max() / np.abs(Wo).max() <= 1e-4


@pytest.mark.parametrize("d,H,slots_per_sm", [(32, 4, 12), (16, 16, 16)])
def test_missing_chunk_wrap_schedule(short_waits, d, H, slots_per_sm):
    """The d = 32 and d = 16 kernels on the wrap-around schedule (more streams
    than warp slots): a missing chunk ends every slot with the timeout status,
    also the slots whose next piece's chunks were already issued, and the next
    call is correct."""
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    B = (slots_per_sm * n_sm) // H + 7
    wl = inputs.Workload("t", B, 100, H, d, 1, True, 77 + d, "normal")
    x, W0 = inputs.make_inputs(wl)
    xd, W0d = torch.from_numpy(x).to(DEV), torch.from_numpy(W0).to(DEV)
    assert binding.srwm_last_device_status() == 0

    binding.srwm_debug_skip_x_chunk(1)
    binding.srwm_forward_balanced(xd, W0d, 1, True)
    assert binding.srwm_last_device_status() == binding.SRWM_ERR_TIMEOUT
    assert binding.srwm_last_device_status() == 0

    binding.srwm_debug_skip_x_chunk(-1)
    y, Wf = binding.srwm_forward_balanced(xd, W0d, 1, True)
    assert binding.srwm_last_device_status() == 0
    rng = np.random.default_rng(3)
    for b in sorted(set(int(v) for v in rng.integers(0, B, 6)) | {0, B - 1}):
        yo, Wo = oracle.forward(x[b:b + 1], W0, 1, True)
        assert np.abs(y[b].cpu().numpy() - yo[0]).max() / np.abs(yo).max() <= 1e-4
        assert np.abs(Wf[b].cpu().numpy() - Wo[0]).max() / np.abs(Wo).max() <= 1e-4
