"""srwm_forward_balanced_noalloc: the balanced schedule for callers that
cannot allocate device memory (its scratch is a fixed array inside the
library).  This file is collected last on purpose.

Checked through the C ABI on two calls in a row (the second call finds the
counters the first one left behind):
  * with short forced segments, so the segment schedule's counters are used;
  * on the wrap-around schedule (d = 32, more streams than warp slots, no
    forced segments), which zeroes and reads the same array;
each time against srwm_forward_balanced with a caller-made workspace and
against the oracle.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from self_referential_weight_gb300 import binding, inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _lib():
    lib = binding._lib()
    P, I = ctypes.c_void_p, ctypes.c_int
    lib.srwm_forward_balanced_noalloc.argtypes = [P, P, I, I, I, I, I, I, P, P, P]
    lib.srwm_forward_balanced_noalloc.restype = I
    return lib


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def rel(a, b):
    return float(np.abs(np.asarray(a, np.float64) - b).max() / max(np.abs(b).max(), 1e-30))


def _two_calls(wl):
    """Two no-alloc calls in a row, each checked against srwm_forward_balanced
    (bitwise: same kernels, same schedule) and against the oracle."""
    lib = _lib()
    x_np, W0_np = inputs.make_inputs(wl)
    x, W0 = torch.from_numpy(x_np).to(DEV), torch.from_numpy(W0_np).to(DEV)
    yo, Wo = oracle.forward(x_np, W0_np, wl.n_lr, wl.softmax_input)
    stream = torch.cuda.current_stream()
    for call in range(2):
        y = torch.full(x.shape, float("nan"), device=DEV)
        Wf = torch.full((wl.B, wl.H, wl.m, wl.d), float("nan"), device=DEV)
        rc = lib.srwm_forward_balanced_noalloc(_ptr(x), _ptr(W0), wl.B, wl.T, wl.H, wl.d, wl.n_lr,
                                               int(wl.softmax_input), _ptr(y), _ptr(Wf),
                                               ctypes.c_void_p(stream.cuda_stream))
        assert rc == 0, binding.srwm_status_string(rc)
        yr, Wr = binding.srwm_forward_balanced(x, W0, wl.n_lr, wl.softmax_input)
        torch.cuda.synchronize()
        assert binding.srwm_last_device_status() == 0
        got_y, got_w = y.cpu().numpy(), Wf.cpu().numpy()
        assert np.isfinite(got_y).all() and np.isfinite(got_w).all(), f"call {call}: outputs not fully written"
        np.testing.assert_array_equal(got_y, yr.cpu().numpy(), err_msg=f"call {call}")
        np.testing.assert_array_equal(got_w, Wr.cpu().numpy(), err_msg=f"call {call}")
        for b in range(wl.B):
            assert rel(got_y[b], yo[b]) <= 1e-4 and rel(got_w[b], Wo[b]) <= 1e-4, (call, b)


@pytest.mark.parametrize("d,n_lr,smx", [(64, 4, False), (32, 1, True), (16, 4, False)])
def test_noalloc_forced_segments_two_calls(d, n_lr, smx):
    binding.srwm_debug_set_segment_len(32)
    try:
        _two_calls(inputs.Workload("t", 3, 150, 2, d, n_lr, smx, 200 + d, "normal"))
    finally:
        binding.srwm_debug_set_segment_len(0)


@pytest.mark.parametrize("n_lr,smx", [(1, True), (4, False)])
def test_noalloc_wrap_schedule_two_calls(n_lr, smx):
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    H = 4
    B = (12 * n_sm) // H + 7   # 12 warp slots per SM at d = 32: 28 more streams than slots
    _two_calls(inputs.Workload("t", B, 70, H, 32, n_lr, smx, 260 + n_lr, "normal"))


def test_noalloc_rejects_more_streams_than_its_array():
    lib = _lib()
    x = torch.zeros(16, device=DEV)
    rc = lib.srwm_forward_balanced_noalloc(_ptr(x), _ptr(x), 65537, 1, 1, 16, 4, 0, _ptr(x), _ptr(x), None)
    assert rc == 2   # SRWM_ERR_SHAPE, before anything is enqueued
