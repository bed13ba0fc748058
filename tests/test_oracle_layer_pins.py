"""Pins of the layer oracle (oracle/srwm_layer.py), no GPU.

  * LN on a hand-computed row: [1, 2, 3, 4] has mean 2.5 and biased variance
    1.25, so LN = (v - 2.5) / sqrt(1.25 + 1e-5), then the per-feature affine map;
  * LN invariants: zero mean and variance var / (var + eps) per token;
  * W0 = 0 and W1 = 0: the SRWM output is zero (pin c2) and the feed-forward
    block is ReLU(b1) W2^T + b2, so out = u + ReLU(b1) W2^T + b2 exactly;
  * a closed ReLU (b1 = -1e3): the feed-forward block is b2, so out - b2 is
    u + the SRWM oracle's output on LN1(u) -- the wiring LN1 -> SRWM ->
    residual against the pinned SRWM oracle;
  * brute force: explicit loops over tokens and features on a tiny layer.
Sources: "Metalearning Continual Learning Algorithms", section 2.3; the review
"SRWM:让权重矩阵学习修改自身", section 2.4.
"""
import numpy as np

import oracle
from oracle import srwm_layer
from self_referential_weight_gb300 import inputs


def _params(H, d, n_lr, d_ff, seed):
    return inputs.make_layer_params(H, d, n_lr, d_ff, seed)


def test_layer_norm_hand_row():
    v = np.array([[1.0, 2.0, 3.0, 4.0]])
    g = np.array([1.0, 2.0, 0.5, -1.0])
    b = np.array([0.0, 1.0, -1.0, 0.25])
    s = np.sqrt(1.25 + 1e-5)
    expect = np.array([[-1.5 / s, 2 * (-0.5 / s) + 1.0, 0.5 * (0.5 / s) - 1.0, -(1.5 / s) + 0.25]])
    np.testing.assert_allclose(srwm_layer.layer_norm(v, g, b), expect, rtol=0, atol=1e-15)


def test_layer_norm_invariants():
    rng = np.random.default_rng(3)
    v = rng.standard_normal((5, 7, 48)) * 3.0 + 2.0
    o = srwm_layer.layer_norm(v, np.ones(48), np.zeros(48))
    np.testing.assert_allclose(o.mean(-1), 0.0, atol=1e-14)
    var = v.var(-1)
    np.testing.assert_allclose(o.var(-1), var / (var + 1e-5), rtol=1e-12)


def test_zero_state_and_zero_first_weight():
    H, d, n_lr, d_ff = 2, 16, 4, 64
    p = _params(H, d, n_lr, d_ff, 5)
    p["W0"] = np.zeros_like(p["W0"])
    p["W1"] = np.zeros_like(p["W1"])
    u = inputs.make_layer_input(2, 9, H * d, 5)
    out, Wf = srwm_layer.layer_forward(u, H, n_lr, False, p)
    assert not Wf.any()
    ff = np.maximum(p["b1"].astype(np.float64), 0) @ p["W2"].astype(np.float64).T + p["b2"]
    np.testing.assert_allclose(out, u.astype(np.float64) + ff, rtol=0, atol=1e-12)


def test_closed_relu_exposes_srwm_wiring():
    H, d, n_lr, d_ff = 2, 32, 1, 64
    p = _params(H, d, n_lr, d_ff, 6)
    p["b1"] = np.full_like(p["b1"], -1e3)
    u = inputs.make_layer_input(3, 11, H * d, 6)
    out, Wf = srwm_layer.layer_forward(u, H, n_lr, True, p)
    a = srwm_layer.layer_norm(u, p["ln1_gamma"], p["ln1_beta"]).astype(np.float32).reshape(3, 11, H, d)
    y, Wo = oracle.forward(a, p["W0"], n_lr, True)
    np.testing.assert_allclose(out - p["b2"], u + y.reshape(3, 11, H * d), rtol=0, atol=1e-12)
    np.testing.assert_array_equal(Wf, Wo)


def test_brute_force_tiny_layer():
    H, d, n_lr, d_ff = 1, 16, 4, 8
    p = _params(H, d, n_lr, d_ff, 7)
    u = inputs.make_layer_input(1, 3, H * d, 7).astype(np.float64)
    out, _ = srwm_layer.layer_forward(u, H, n_lr, False, p)
    B, T, D = u.shape
    g1, be1, g2, be2 = (p[k].astype(np.float64) for k in ("ln1_gamma", "ln1_beta", "ln2_gamma", "ln2_beta"))
    W1, b1, W2, b2 = (p[k].astype(np.float64) for k in ("W1", "b1", "W2", "b2"))

    def ln(row, g, be):
        mu = sum(row) / D
        var = sum((x - mu) ** 2 for x in row) / D
        return [(row[i] - mu) / (var + 1e-5) ** 0.5 * g[i] + be[i] for i in range(D)]

    a = np.array([[ln(list(u[b, t]), g1, be1) for t in range(T)] for b in range(B)])
    y, _ = oracle.forward(a.astype(np.float32).reshape(B, T, H, d), p["W0"], n_lr, False)
    y = y.reshape(B, T, D)
    for b in range(B):
        for t in range(T):
            h = [u[b, t, i] + y[b, t, i] for i in range(D)]
            v = ln(h, g2, be2)
            hid = [max(sum(W1[j, i] * v[i] for i in range(D)) + b1[j], 0.0) for j in range(d_ff)]
            for i in range(D):
                expect = h[i] + sum(W2[i, j] * hid[j] for j in range(d_ff)) + b2[i]
                assert abs(out[b, t, i] - expect) <= 1e-12 * max(1.0, abs(expect))
