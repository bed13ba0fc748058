"""Layer oracle (test infrastructure only): one Recursive Self-Transformer layer
in float64 NumPy, step by step.

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may use
it.  The SRWM replaces multi-head self-attention in a Transformer block
("Metalearning Continual Learning Algorithms", section 2.3); the layer norms,
feed-forward block and residual connections stay as in the Transformer (the
review "SRWM:让权重矩阵学习修改自身", section 2.4).  The block order is read as
pre-LN:
    a = LN1(u);  y = SRWM(a);  h = u + y;  out = h + W2 ReLU(W1 LN2(h) + b1) + b2
with LN over the D features of a token (biased variance, eps = 1e-5).  The
SRWM step is the C oracle's (pinned in tests/test_oracle_pins.py); its input
a is rounded to float32 first, as the C oracle takes float32 inputs.
Pinned in tests/test_oracle_layer_pins.py.
"""
import numpy as np

from . import srwm_oracle

LN_EPS = 1e-5


def layer_norm(v, gamma, beta, eps=LN_EPS):
    """(v - mean) / sqrt(var + eps) * gamma + beta over the last axis (float64)."""
    v = np.asarray(v, np.float64)
    mu = v.mean(axis=-1, keepdims=True)
    var = ((v - mu) ** 2).mean(axis=-1, keepdims=True)
    return (v - mu) / np.sqrt(var + eps) * np.asarray(gamma, np.float64) + np.asarray(beta, np.float64)


def feed_forward(v, W1, b1, W2, b2):
    """W2 ReLU(W1 v + b1) + b2 per token (weights in PyTorch Linear layout)."""
    hdn = np.maximum(np.asarray(v, np.float64) @ np.asarray(W1, np.float64).T + np.asarray(b1, np.float64), 0.0)
    return hdn @ np.asarray(W2, np.float64).T + np.asarray(b2, np.float64)


def layer_forward(u, H, n_lr, softmax_input, p, n_threads=None):
    """u [B, T, D] and the parameter dict p (ln1_gamma, ln1_beta, W0, ln2_gamma,
    ln2_beta, W1, b1, W2, b2) -> (out [B, T, D] float64, W_final [B, H, m, d])."""
    u = np.asarray(u, np.float64)
    B, T, D = u.shape
    d = D // H
    a = layer_norm(u, p["ln1_gamma"], p["ln1_beta"])
    y, W_final = srwm_oracle.forward(a.astype(np.float32).reshape(B, T, H, d), p["W0"], n_lr, softmax_input,
                                     n_threads=n_threads)
    h = u + np.asarray(y, np.float64).reshape(B, T, D)
    out = h + feed_forward(layer_norm(h, p["ln2_gamma"], p["ln2_beta"]), p["W1"], p["b1"], p["W2"], p["b2"])
    return out, W_final
