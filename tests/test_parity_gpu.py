"""GPU parity: the sm_103a library against the CPU oracle, element by element,
on the same seeded inputs.

Tolerance (fp32 state and arithmetic against the float64 oracle):
    max|gpu - oracle| / max|oracle| <= 1e-4 for T <= 1024, <= 1e-3 up to T = 8192,
for y and for W_final alike.  The oracle's own fp32 floor on these workloads is
<= 5e-6 (tests/test_oracle_pins.py::test_c8_fp32_floor).
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from self_referential_weight_gb300 import binding, inputs

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def tol(T):
    return 1e-4 if T <= 1024 else 1e-3


def rel(a, b):
    return float(np.abs(np.asarray(a, np.float64) - b).max() / max(np.abs(b).max(), 1e-30))


def run_gpu(x, W0, n_lr, smx):
    y, Wf = binding.srwm_forward(torch.from_numpy(x).to(DEV), torch.from_numpy(W0).to(DEV), n_lr, smx)
    torch.cuda.synchronize()
    assert binding.srwm_last_device_status() == 0
    return y.cpu().numpy(), Wf.cpu().numpy()


# ------------------------------------------------------------------ small shapes
# Several TMA chunks (16 steps for d <= 32, 32 for d = 64) plus a ragged tail,
# and stream counts that leave the last CTA partly empty.
@pytest.mark.parametrize("d", [16, 32, 64])
@pytest.mark.parametrize("n_lr", [1, 4])
@pytest.mark.parametrize("smx", [False, True])
def test_small_all_variants(d, n_lr, smx):
    wl = inputs.Workload("t", 3, 75, 3, d, n_lr, smx, 10 + d + n_lr + smx, "normal")
    x, W0 = inputs.make_inputs(wl)
    y, Wf = run_gpu(x, W0, n_lr, smx)
    yo, Wo = oracle.forward(x, W0, n_lr, smx)
    assert rel(y, yo) <= 1e-4
    assert rel(Wf, Wo) <= 1e-4


@pytest.mark.parametrize("d", [16, 32, 64])
@pytest.mark.parametrize("T", [1, 2, 15, 16, 17, 31, 32, 33, 64])
def test_step_count_edges(d, T):
    wl = inputs.Workload("t", 2, T, 5, d, 4, False, 100 + T, "normal")
    x, W0 = inputs.make_inputs(wl)
    y, Wf = run_gpu(x, W0, 4, False)
    yo, Wo = oracle.forward(x, W0, 4, False)
    assert rel(y, yo) <= 1e-4 and rel(Wf, Wo) <= 1e-4


@pytest.mark.parametrize("d", [16, 32, 64])
def test_zero_steps_copies_W0(d):
    W0 = inputs.make_W0(3, d, 4, seed=5)
    x = torch.empty((2, 0, 3, d), device=DEV)
    y, Wf = binding.srwm_forward(x, torch.from_numpy(W0).to(DEV), 4)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(Wf.cpu().numpy(), np.broadcast_to(W0, (2,) + W0.shape))


@pytest.mark.parametrize("d", [16, 32, 64])
def test_zero_matrix_stays_zero(d):
    """The W0 = 0 fixed point holds exactly on the GPU too."""
    wl = inputs.Workload("t", 2, 40, 2, d, 4, False, 7, "normal")
    x = inputs.make_x(wl)
    W0 = np.zeros((2, 3 * d + 4, d), np.float32)
    y, Wf = run_gpu(x, W0, 4, False)
    assert not y.any() and not Wf.any()


@pytest.mark.parametrize("n_streams", [1, 5, 6, 7, 8, 9, 13, 17])
def test_stream_counts_fill_ctas(n_streams):
    """Streams per CTA are 8 (d=16) and 6 (d=32): counts around those."""
    for d in (16, 32):
        wl = inputs.Workload("t", n_streams, 20, 1, d, 4, False, n_streams, "normal")
        x, W0 = inputs.make_inputs(wl)
        y, Wf = run_gpu(x, W0, 4, False)
        yo, Wo = oracle.forward(x, W0, 4, False)
        assert rel(y, yo) <= 1e-4 and rel(Wf, Wo) <= 1e-4


# ------------------------------------------------------------------ named workloads
def test_tiny_full():
    wl = inputs.workload("tiny")
    x, W0 = inputs.make_inputs(wl)
    y, Wf = run_gpu(x, W0, wl.n_lr, wl.softmax_input)
    yo, Wo = oracle.forward(x, W0, wl.n_lr, wl.softmax_input)
    assert rel(y, yo) <= tol(wl.T) and rel(Wf, Wo) <= tol(wl.T)


def test_fewshot_full():
    wl = inputs.workload("fewshot")
    x, W0 = inputs.make_inputs(wl)
    y, Wf = run_gpu(x, W0, wl.n_lr, wl.softmax_input)
    yo, Wo = oracle.forward(x, W0, wl.n_lr, wl.softmax_input)
    assert rel(y, yo) <= tol(wl.T) and rel(Wf, Wo) <= tol(wl.T)


def per_stream_rel(got, ref, T):
    """Largest per-(b, h) relative error of y [B,T,H,d] and W_final [B,H,m,d]."""
    B, _, H, _ = ref[0].shape
    worst_y = worst_w = 0.0
    for b in range(B):
        for h in range(H):
            worst_y = max(worst_y, rel(got[0][b, :, h], ref[0][b, :, h]))
            worst_w = max(worst_w, rel(got[1][b, h], ref[1][b, h]))
    return worst_y, worst_w


@pytest.mark.parametrize("name", ["mid", "long", "rl", "fewshot"])
def test_full_size_every_stream(name):
    """Full-size workloads, every (b, h) stream against the oracle, for both the
    plain launch (srwm_forward) and the launch the benchmark times
    (srwm_forward_balanced: one wave on mid and long, the wrap-around schedule
    on rl).  The bar holds over the whole tensor and for each stream alone."""
    wl = inputs.workload(name)
    x, W0 = inputs.make_inputs(wl)
    yo, Wo = oracle.forward(x, W0, wl.n_lr, wl.softmax_input)
    xd, W0d = torch.from_numpy(x).to(DEV), torch.from_numpy(W0).to(DEV)
    for launch in ("plain", "balanced"):
        if launch == "plain":
            y, Wf = binding.srwm_forward(xd, W0d, wl.n_lr, wl.softmax_input)
        else:
            y, Wf = binding.srwm_forward_balanced(xd, W0d, wl.n_lr, wl.softmax_input)
        torch.cuda.synchronize()
        assert binding.srwm_last_device_status() == 0
        y, Wf = y.cpu().numpy(), Wf.cpu().numpy()
        ey, ew = rel(y, yo), rel(Wf, Wo)
        assert ey <= tol(wl.T) and ew <= tol(wl.T), (launch, ey, ew)
        sy, sw = per_stream_rel((y, Wf), (yo, Wo), wl.T)
        assert sy <= tol(wl.T) and sw <= tol(wl.T), (launch, sy, sw)
        del y, Wf


# ------------------------------------------------------------------ structure
@pytest.mark.parametrize("d", [16, 32, 64])
def test_stream_slice_is_bitwise_equal(d):
    """Streams are independent: running one (b, h) alone gives the same bits."""
    wl = inputs.Workload("t", 3, 50, 4, d, 4, False, 21, "normal")
    x, W0 = inputs.make_inputs(wl)
    y, Wf = run_gpu(x, W0, 4, False)
    for b, h in [(0, 0), (2, 3), (1, 2)]:
        ys, Wfs = run_gpu(np.ascontiguousarray(x[b:b + 1, :, h:h + 1]), W0[h:h + 1], 4, False)
        np.testing.assert_array_equal(ys[0, :, 0], y[b, :, h])
        np.testing.assert_array_equal(Wfs[0, 0], Wf[b, h])


@pytest.mark.parametrize("d", [16, 32, 64])
def test_deterministic(d):
    wl = inputs.Workload("t", 4, 70, 3, d, 1, True, 22, "normal")
    x, W0 = inputs.make_inputs(wl)
    a = run_gpu(x, W0, 1, True)
    b = run_gpu(x, W0, 1, True)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


@pytest.mark.parametrize("d", [16, 32, 64])
@pytest.mark.parametrize("n_lr,smx", [(4, False), (1, True)])
def test_step_matches_oracle_and_chains_to_forward(d, n_lr, smx):
    """srwm_step from per-sequence states equals the oracle's one step; T
    chained steps (in place) equal one srwm_forward call."""
    wl = inputs.Workload("t", 3, 12, 2, d, n_lr, smx, 30 + d, "normal")
    x, W0 = inputs.make_inputs(wl)
    m = wl.m
    # one step from distinct per-sequence states
    Wseq = (W0[None] + 0.05 * np.random.default_rng(1).standard_normal((3, 2, m, d))).astype(np.float32)
    yt, Wo = binding.srwm_step(torch.from_numpy(np.ascontiguousarray(x[:, 0])).to(DEV),
                               torch.from_numpy(Wseq).to(DEV), n_lr, smx)
    torch.cuda.synchronize()
    yo, Woo = oracle.forward(x[:, :1], Wseq, n_lr, smx, per_sequence=True)
    assert rel(yt.cpu().numpy(), yo[:, 0]) <= 1e-5
    assert rel(Wo.cpu().numpy(), Woo) <= 1e-5
    # chained in place
    W = torch.from_numpy(np.ascontiguousarray(np.broadcast_to(W0, (3, 2, m, d)))).to(DEV)
    ys = []
    for t in range(wl.T):
        yt, _ = binding.srwm_step(torch.from_numpy(np.ascontiguousarray(x[:, t])).to(DEV), W, n_lr, smx,
                                  W_out=W)
        ys.append(yt.cpu().numpy())
    y_chain = np.stack(ys, axis=1)
    y, Wf = run_gpu(x, W0, n_lr, smx)
    assert rel(y_chain, y) <= 1e-5
    assert rel(W.cpu().numpy(), Wf) <= 1e-5


# ------------------------------------------------------------------ boundary on a GPU
def test_host_pointer_is_rejected():
    lib = binding._lib()
    x = torch.zeros((1, 4, 1, 16))           # host memory
    W0 = torch.zeros((1, 52, 16), device=DEV)
    y = torch.zeros((1, 4, 1, 16), device=DEV)
    Wf = torch.zeros((1, 1, 52, 16), device=DEV)
    rc = lib.srwm_forward(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(W0.data_ptr()), 1, 4, 1, 16,
                          4, 0, ctypes.c_void_p(y.data_ptr()), ctypes.c_void_p(Wf.data_ptr()), None)
    assert rc == 8


def test_device_alias_is_rejected():
    buf = torch.zeros(4096, device=DEV)
    lib = binding._lib()
    p = buf.data_ptr()
    rc = lib.srwm_forward(ctypes.c_void_p(p), ctypes.c_void_p(p + 8192), 1, 4, 1, 16, 4, 0,
                          ctypes.c_void_p(p + 64), ctypes.c_void_p(p + 12288), None)
    assert rc == 5


def test_binding_raises_on_error():
    x = torch.zeros((1, 4, 1, 48), device=DEV)
    W0 = torch.zeros((1, 148, 48), device=DEV)
    with pytest.raises(binding.SrwmError) as e:
        binding.srwm_forward(x, W0, 4)
    assert e.value.status == 3


@pytest.mark.parametrize("n_lr,smx", [(4, False), (1, True)])
def test_d64_more_streams_than_sms(n_lr, smx):
    """d = 64 with more (b, h) streams than SMs (the four-warp-per-stream
    variant; fewer streams use eight warps each), checked in full."""
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    B = n_sm // 8 + 3
    wl = inputs.Workload("t", B, 40, 8, 64, n_lr, smx, 77, "normal")
    x, W0 = inputs.make_inputs(wl)
    y, Wf = run_gpu(x, W0, n_lr, smx)
    yo, Wo = oracle.forward(x, W0, n_lr, smx)
    assert rel(y, yo) <= 1e-4 and rel(Wf, Wo) <= 1e-4


def many_stream_batch(n_sm):
    """B for H = 8 streams per sequence so that d = 64 runs more than two
    streams per SM (the two-warp kernel), with a partly filled last wave."""
    return (2 * n_sm) // 8 + 3


@pytest.mark.parametrize("n_lr", [1, 4])
@pytest.mark.parametrize("smx", [False, True])
def test_d64_many_streams_all_variants(n_lr, smx):
    """More than two d = 64 streams per SM selects two warps per stream (four
    CTAs per SM); checked in full against the oracle over several TMA chunks
    and a ragged tail."""
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    wl = inputs.Workload("t", many_stream_batch(n_sm), 75, 8, 64, n_lr, smx, 130 + n_lr + smx, "normal")
    x, W0 = inputs.make_inputs(wl)
    y, Wf = run_gpu(x, W0, n_lr, smx)
    yo, Wo = oracle.forward(x, W0, n_lr, smx)
    assert rel(y, yo) <= 1e-4 and rel(Wf, Wo) <= 1e-4


@pytest.mark.parametrize("T", [1, 31, 32, 33, 64])
def test_d64_many_streams_step_edges(T):
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    wl = inputs.Workload("t", many_stream_batch(n_sm), T, 8, 64, 4, False, 140 + T, "normal")
    x, W0 = inputs.make_inputs(wl)
    y, Wf = run_gpu(x, W0, 4, False)
    yo, Wo = oracle.forward(x, W0, 4, False)
    assert rel(y, yo) <= 1e-4 and rel(Wf, Wo) <= 1e-4


def test_d64_many_streams_slice_and_determinism():
    """A stream computed alone (four-warp kernel) equals the same stream in a
    many-stream batch (two-warp kernel) within fp32 rounding; the batch is
    bitwise repeatable."""
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    wl = inputs.Workload("t", many_stream_batch(n_sm), 70, 8, 64, 4, False, 150, "normal")
    x, W0 = inputs.make_inputs(wl)
    y, Wf = run_gpu(x, W0, 4, False)
    y2, Wf2 = run_gpu(x, W0, 4, False)
    np.testing.assert_array_equal(y, y2)
    np.testing.assert_array_equal(Wf, Wf2)
    b, h = wl.B - 2, 5
    ys, Ws = run_gpu(np.ascontiguousarray(x[b:b + 1, :, h:h + 1]), np.ascontiguousarray(W0[h:h + 1]), 4, False)
    assert rel(y[b, :, h], ys[0, :, 0]) <= 1e-5 and rel(Wf[b, h], Ws[0, 0]) <= 1e-5


def test_d64_many_streams_step_chains_to_forward():
    """srwm_step over many per-sequence states (two-warp kernel, T = 1),
    chained in place, equals srwm_forward."""
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    wl = inputs.Workload("t", many_stream_batch(n_sm), 9, 8, 64, 4, True, 160, "normal")
    x, W0 = inputs.make_inputs(wl)
    y, Wf = run_gpu(x, W0, 4, True)
    xd = torch.from_numpy(x).to(DEV)
    W = torch.from_numpy(np.ascontiguousarray(np.broadcast_to(W0, (wl.B,) + W0.shape))).to(DEV)
    ys = []
    for t in range(wl.T):
        yt, W = binding.srwm_step(xd[:, t].contiguous(), W, 4, True, W_out=W)
        ys.append(yt.cpu().numpy())
    torch.cuda.synchronize()
    assert binding.srwm_last_device_status() == 0
    assert rel(np.stack(ys, axis=1), y) <= 1e-5 and rel(W.cpu().numpy(), Wf) <= 1e-5


@pytest.mark.parametrize("d", [16, 32, 64])
@pytest.mark.parametrize("n_lr,smx", [(4, False), (1, True)])
def test_forward_from_resumes_a_split_sequence(d, n_lr, smx):
    """State carry: T1 steps of srwm_forward, then T - T1 steps of
    srwm_forward_from on the returned state (in place), equal one call over T
    steps; the second window also matches the oracle started from its state."""
    wl = inputs.Workload("t", 3, 70, 2, d, n_lr, smx, 90 + d, "normal")
    x, W0 = inputs.make_inputs(wl)
    T1 = 37
    y_full, Wf_full = run_gpu(x, W0, n_lr, smx)
    xd = torch.from_numpy(x).to(DEV)
    y1, W = binding.srwm_forward(xd[:, :T1].contiguous(), torch.from_numpy(W0).to(DEV), n_lr, smx)
    W_mid = W.cpu().numpy()
    y2, W = binding.srwm_forward_from(xd[:, T1:].contiguous(), W, n_lr, smx, W_final=W)
    torch.cuda.synchronize()
    assert binding.srwm_last_device_status() == 0
    y_split = np.concatenate([y1.cpu().numpy(), y2.cpu().numpy()], axis=1)
    assert rel(y_split, y_full) <= 1e-5
    assert rel(W.cpu().numpy(), Wf_full) <= 1e-5
    yo, Wo = oracle.forward(np.ascontiguousarray(x[:, T1:]), W_mid, n_lr, smx, per_sequence=True)
    assert rel(y2.cpu().numpy(), yo) <= 1e-4 and rel(W.cpu().numpy(), Wo) <= 1e-4


def test_forward_from_zero_steps_copies_state():
    W = torch.randn(2, 3, 52, 16, device=DEV)
    x = torch.empty((2, 0, 3, 16), device=DEV)
    _, Wf = binding.srwm_forward_from(x, W, 4)
    torch.cuda.synchronize()
    assert torch.equal(Wf, W)


@pytest.mark.parametrize("d", [16, 32, 64])
@pytest.mark.parametrize("n_lr,smx", [(4, False), (1, True)])
def test_balanced_forced_segments_match(d, n_lr, smx):
    """The balanced schedule with short forced segments (32 steps, a ragged
    last one): every stream hops between slots through W_final and the
    progress counters.  Equals srwm_forward within fp32 rounding, matches the
    oracle, and is deterministic."""
    wl = inputs.Workload("t", 3, 150, 2, d, n_lr, smx, 120 + d, "normal")
    x, W0 = inputs.make_inputs(wl)
    y, Wf = run_gpu(x, W0, n_lr, smx)
    xd, W0d = torch.from_numpy(x).to(DEV), torch.from_numpy(W0).to(DEV)
    binding.srwm_debug_set_segment_len(32)
    try:
        yb, Wb = binding.srwm_forward_balanced(xd, W0d, n_lr, smx)
        yb2, Wb2 = binding.srwm_forward_balanced(xd, W0d, n_lr, smx)
        torch.cuda.synchronize()
        assert binding.srwm_last_device_status() == 0
    finally:
        binding.srwm_debug_set_segment_len(0)
    yb, Wb = yb.cpu().numpy(), Wb.cpu().numpy()
    assert rel(yb, y) <= 1e-5 and rel(Wb, Wf) <= 1e-5
    np.testing.assert_array_equal(yb, yb2.cpu().numpy())
    np.testing.assert_array_equal(Wb, Wb2.cpu().numpy())
    yo, Wo = oracle.forward(x, W0, n_lr, smx)
    assert rel(yb, yo) <= 1e-4 and rel(Wb, Wo) <= 1e-4


@pytest.mark.parametrize("n_lr,smx", [(4, False), (1, True)])
def test_balanced_forced_segments_many_streams(n_lr, smx):
    """The balanced schedule on the two-warp d = 64 kernel: more streams than
    its slots' worth per wave, forced 32-step segments."""
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    wl = inputs.Workload("t", (5 * n_sm) // 8 + 1, 100, 8, 64, n_lr, smx, 170 + n_lr, "normal")
    x, W0 = inputs.make_inputs(wl)
    y, Wf = run_gpu(x, W0, n_lr, smx)
    xd, W0d = torch.from_numpy(x).to(DEV), torch.from_numpy(W0).to(DEV)
    binding.srwm_debug_set_segment_len(32)
    try:
        yb, Wb = binding.srwm_forward_balanced(xd, W0d, n_lr, smx)
        torch.cuda.synchronize()
        assert binding.srwm_last_device_status() == 0
    finally:
        binding.srwm_debug_set_segment_len(0)
    yb, Wb = yb.cpu().numpy(), Wb.cpu().numpy()
    assert rel(yb, y) <= 1e-5 and rel(Wb, Wf) <= 1e-5
    yo, Wo = oracle.forward(x, W0, n_lr, smx)
    assert rel(yb, yo) <= 1e-4 and rel(Wb, Wo) <= 1e-4


@pytest.mark.parametrize("T", [70, 64, 1])
@pytest.mark.parametrize("n_lr,smx", [(1, True), (4, False)])
@pytest.mark.parametrize("d,H,slots_per_sm", [(32, 4, 12), (16, 16, 16)])
def test_balanced_wrap_schedule(d, H, slots_per_sm, T, n_lr, smx):
    """The d = 32 and d = 16 kernels' wrap-around schedule: more streams than
    warp slots, each slot an equal range of all streams' steps.  T = 70 puts
    the split points inside TMA chunks; T = 1 never splits.  Every stream is
    checked against the plain launch and the oracle; results are
    deterministic."""
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    B = (slots_per_sm * n_sm) // H + 7   # warp slots per SM: 12 (d = 32), 16 (d = 16)
    wl = inputs.Workload("t", B, T, H, d, n_lr, smx, 300 + T + n_lr + d, "normal")
    x, W0 = inputs.make_inputs(wl)
    y, Wf = run_gpu(x, W0, n_lr, smx)
    xd, W0d = torch.from_numpy(x).to(DEV), torch.from_numpy(W0).to(DEV)
    yb, Wb = binding.srwm_forward_balanced(xd, W0d, n_lr, smx)
    yb2, Wb2 = binding.srwm_forward_balanced(xd, W0d, n_lr, smx)
    torch.cuda.synchronize()
    assert binding.srwm_last_device_status() == 0
    yb, Wb = yb.cpu().numpy(), Wb.cpu().numpy()
    assert rel(yb, y) <= 1e-5 and rel(Wb, Wf) <= 1e-5
    np.testing.assert_array_equal(yb, yb2.cpu().numpy())
    np.testing.assert_array_equal(Wb, Wb2.cpu().numpy())
    yo, Wo = oracle.forward(x, W0, n_lr, smx)
    for b in range(B):
        assert rel(yb[b], yo[b]) <= 1e-4 and rel(Wb[b], Wo[b]) <= 1e-4
