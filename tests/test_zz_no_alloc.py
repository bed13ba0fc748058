"""srwm_forward_balanced_noalloc: the balanced schedule for callers that
cannot allocate device memory (its scratch is a fixed array inside the
library).  This file is collected last on purpose.

Checked through the C ABI against srwm_forward_balanced with a caller-made
workspace, on two calls in a row (the second call finds the counters the
first one left behind), with short forced segments so the counters are used.
"""
import ctypes

import numpy as np
import pytest
import torch

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


@pytest.mark.parametrize("d,n_lr,smx", [(64, 4, False), (32, 1, True), (16, 4, False)])
def test_noalloc_matches_balanced_on_two_calls(d, n_lr, smx):
    lib = _lib()
    wl = inputs.Workload("t", 3, 150, 2, d, n_lr, smx, 200 + d, "normal")
    x_np, W0_np = inputs.make_inputs(wl)
    x, W0 = torch.from_numpy(x_np).to(DEV), torch.from_numpy(W0_np).to(DEV)
    stream = torch.cuda.current_stream()
    binding.srwm_debug_set_segment_len(32)
    try:
        for call in range(2):
            y = torch.full(x.shape, float("nan"), device=DEV)
            Wf = torch.full((wl.B, wl.H, wl.m, wl.d), float("nan"), device=DEV)
            rc = lib.srwm_forward_balanced_noalloc(_ptr(x), _ptr(W0), wl.B, wl.T, wl.H, wl.d, n_lr, int(smx),
                                                   _ptr(y), _ptr(Wf), ctypes.c_void_p(stream.cuda_stream))
            assert rc == 0, binding.srwm_status_string(rc)
            yr, Wr = binding.srwm_forward_balanced(x, W0, n_lr, smx)
            torch.cuda.synchronize()
            assert binding.srwm_last_device_status() == 0
            for got, ref in ((y, yr), (Wf, Wr)):
                got, ref = got.cpu().numpy(), ref.cpu().numpy()
                assert np.isfinite(got).all(), f"call {call}: outputs not fully written"
                assert np.abs(got - ref).max() <= 1e-5 * np.abs(ref).max(), f"call {call}"
    finally:
        binding.srwm_debug_set_segment_len(0)


def test_noalloc_rejects_more_streams_than_its_array():
    lib = _lib()
    x = torch.zeros(16, device=DEV)
    rc = lib.srwm_forward_balanced_noalloc(_ptr(x), _ptr(x), 65537, 1, 1, 16, 4, 0, _ptr(x), _ptr(x), None)
    assert rc == 2   # SRWM_ERR_SHAPE, before anything is enqueued
