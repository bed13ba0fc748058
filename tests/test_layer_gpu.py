"""GPU parity of srwm_layer_forward (one Recursive Self-Transformer layer)
against the float64 layer oracle, on the same seeded inputs and parameters.

Tolerance: max|gpu - oracle| / max|oracle| <= 1e-4 for out, as for the SRWM's
own outputs at these lengths.  The layer norms and the fp32 GEMMs (K <= 4D)
add errors of order 1e-6 on top.
"""
import numpy as np
import pytest
import torch

from oracle import srwm_layer
from self_referential_weight_gb300 import binding, inputs

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def rel(a, b):
    return float(np.abs(np.asarray(a, np.float64) - b).max() / max(np.abs(b).max(), 1e-30))


def run_layer(u, H, n_lr, smx, p, with_state=True):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    B, T, D = u.shape
    d = D // H
    Wf = torch.empty((B, H, 3 * d + n_lr, d), device=DEV) if with_state else None
    out, Wf = binding.srwm_layer_forward(t(u), H, n_lr, smx, t(p["ln1_gamma"]), t(p["ln1_beta"]), t(p["W0"]),
                                         t(p["ln2_gamma"]), t(p["ln2_beta"]), t(p["W1"]), t(p["b1"]), t(p["W2"]),
                                         t(p["b2"]), W_final=Wf)
    torch.cuda.synchronize()
    assert binding.srwm_last_device_status() == 0
    return out.cpu().numpy(), (Wf.cpu().numpy() if Wf is not None else None)


@pytest.mark.parametrize("d", [16, 32, 64])
@pytest.mark.parametrize("n_lr,smx", [(4, False), (1, True)])
def test_layer_matches_oracle(d, n_lr, smx):
    B, T, H = 2, 70, 2
    D = H * d
    p = inputs.make_layer_params(H, d, n_lr, 4 * D, 200 + d + n_lr)
    u = inputs.make_layer_input(B, T, D, 200 + d)
    out, Wf = run_layer(u, H, n_lr, smx, p)
    oo, Wo = srwm_layer.layer_forward(u, H, n_lr, smx, p)
    assert rel(out, oo) <= 1e-4
    assert rel(Wf, Wo) <= 1e-4


def test_layer_wide_model_many_streams():
    """D = 512 (eight heads of 64), 48 sequences: 384 streams, the two-warp
    SRWM kernel, and GEMMs with K = 512 and 2048."""
    B, T, H, d, n_lr = 48, 40, 8, 64, 4
    p = inputs.make_layer_params(H, d, n_lr, 4 * H * d, 210)
    u = inputs.make_layer_input(B, T, H * d, 210)
    out, Wf = run_layer(u, H, n_lr, False, p)
    oo, Wo = srwm_layer.layer_forward(u, H, n_lr, False, p)
    assert rel(out, oo) <= 1e-4 and rel(Wf, Wo) <= 1e-4


def test_layer_without_state_output_and_deterministic():
    B, T, H, d = 3, 33, 4, 32
    p = inputs.make_layer_params(H, d, 1, 256, 220)
    u = inputs.make_layer_input(B, T, H * d, 220)
    a, _ = run_layer(u, H, 1, True, p, with_state=False)
    b, _ = run_layer(u, H, 1, True, p, with_state=False)
    np.testing.assert_array_equal(a, b)


def test_layer_zero_steps_returns_W0():
    H, d = 2, 16
    p = inputs.make_layer_params(H, d, 4, 64, 230)
    u = np.zeros((3, 0, H * d), np.float32)
    _, Wf = run_layer(u, H, 4, False, p)
    np.testing.assert_array_equal(Wf, np.broadcast_to(p["W0"], Wf.shape))


def test_layer_tensor_core_products_agree_with_cublaslt():
    """The default path (this library's tensor-core kernel, bf16 (hi, lo)
    operand pairs) against the cuBLASLt plain-FP32 comparison path and the
    oracle, on the wide shape (D = 512, d_ff = 2048: K = 512 and 2048)."""
    B, T, H, d, n_lr = 16, 40, 8, 64, 4
    p = inputs.make_layer_params(H, d, n_lr, 4 * H * d, 240)
    u = inputs.make_layer_input(B, T, H * d, 240)
    tc, _ = run_layer(u, H, n_lr, False, p)
    binding.srwm_debug_set_layer_gemm(1)
    try:
        ref, _ = run_layer(u, H, n_lr, False, p)
    finally:
        binding.srwm_debug_set_layer_gemm(0)
    oo, _ = srwm_layer.layer_forward(u, H, n_lr, False, p)
    e_tc, e_ref, e_vs = rel(tc, oo), rel(ref, oo), rel(tc, ref)
    print(f"layer out vs oracle: tensor cores {e_tc:.2e}, cuBLASLt FP32 {e_ref:.2e}; between them {e_vs:.2e}")
    assert e_tc <= 1e-4 and e_ref <= 1e-4 and e_vs <= 1e-4


@pytest.mark.parametrize("B,T,H,d,d_ff", [(1, 1, 2, 16, 8), (3, 45, 8, 64, 2048), (2, 33, 2, 32, 24),
                                          (1, 129, 4, 16, 64), (2, 37, 3, 16, 1032)])
def test_layer_tile_edges(B, T, H, d, d_ff):
    """Shapes at the tensor-core products' tile edges: one token, token
    counts off the 128-row tiles, hidden widths below one 256-column tile
    and inner dimensions below one K step (filled with zeros by TMA).  The
    last case takes both K-step configurations at ragged edges: K = 48
    (one 64-wide step, zero-filled), an output width of 1032 (a partial
    256-column tile, 32-column stores clipped), and K = 1032 for the second
    product (32-wide steps, the last one partial)."""
    n_lr = 4
    p = inputs.make_layer_params(H, d, n_lr, d_ff, 250 + T)
    u = inputs.make_layer_input(B, T, H * d, 250 + T)
    out, _ = run_layer(u, H, n_lr, False, p)
    oo, _ = srwm_layer.layer_forward(u, H, n_lr, False, p)
    assert rel(out, oo) <= 1e-4, rel(out, oo)
