"""Pins of the CPU oracle to facts the pages and the mathematics fix.

Each test checks the oracle against something other than itself: the worked
example printed on the review page, an invariant, a closed form, a special case
that reduces to a library routine, or an independent brute-force transcription
on tiny inputs.  A plausible slip anywhere in the oracle (a dropped term, a
wrong sign, a swapped k/q address, a wrong row block, an update applied before
the output is read) fails at least one of them.

Sources:
  [ACL]  "Metalearning Continual Learning Algorithms", section 2.3, Eqs. (1)-(5).
  [REV]  review page "SRWM:让权重矩阵学习修改自身" of "A Modern Self-Referential
         Weight Matrix That Learns to Modify Itself": sections 2.2 (time
         ordering), 2.3 (read-back derivation, norm bound, worked example),
         2.4 (four learning rates, heads), 2.5 (W0 = 0 is a fixed point).
"""
import os

import numpy as np
import pytest
from scipy.special import expit
from scipy.special import softmax as sp_softmax

import oracle
from self_referential_weight_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_example.txt")


def _golden():
    vals = {}
    with open(GOLDEN, encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *rest = line.split()
            vals[key] = np.array([float(v) for v in rest])
    return vals


def _rng(seed):
    return np.random.default_rng(seed)


def _rel(a, b):
    scale = max(np.abs(b).max(), 1e-300)
    return np.abs(np.asarray(a, np.float64) - np.asarray(b, np.float64)).max() / scale


# ---------------------------------------------------------------- c1, c1b
def test_c1_worked_example_delta_update():
    """[REV] 2.3 worked example: w=[1,3], key e1, query e2, eta=0.5 -> [2,3]."""
    g = _golden()
    W = g["w"][None, :]
    assert float(W[0] @ g["phi_k"]) == g["old_value"][0]
    assert float(W[0] @ g["phi_q"]) == g["target_value"][0]
    out = oracle.delta_update(W, g["phi_k"], g["phi_q"], g["eta"])
    np.testing.assert_array_equal(out[0], g["w_updated"])


def test_c1_swapped_addresses_move_the_other_way():
    """With k and q swapped the row moves from 3 towards 1 at address e2."""
    out = oracle.delta_update([[1.0, 3.0]], [0, 1], [1, 0], [0.5])
    np.testing.assert_array_equal(out[0], [1.0, 2.0])


def _c1b_W0():
    # d = 2, one learning rate: m = 3*2 + 1 = 7 rows [o0, o1, k0, k1, q0, q1, beta].
    # With input e1 the key logits are (+40, -40) -> phi(k) ~ e1, the query
    # logits (-40, +40) -> phi(q) ~ e2, and beta = 0 -> gate 0.5.
    return np.array([[[1.0, 3.0], [0.25, -0.5],
                      [40.0, 0.0], [-40.0, 0.0],
                      [-40.0, 0.0], [40.0, 0.0],
                      [0.0, 0.0]]], dtype=np.float32)


def test_c1b_end_to_end_worked_example_and_time_ordering():
    """The worked example through the whole step (Eqs. (1)-(3) with softmax and
    sigmoid), over two steps.  y_0 is read from W_0 (old value 1); y_1 from W_1
    (updated value 2): [REV] 2.2 says the SRWM output uses the pre-update matrix."""
    W0 = _c1b_W0()
    x = np.zeros((1, 2, 1, 2), np.float32)
    x[0, :, 0, 0] = 1.0  # e1 at both steps
    y, Wf = oracle.forward(x, W0, n_lr=1)
    tol = 1e-12
    assert abs(y[0, 0, 0, 0] - 1.0) < tol          # from W_0: row [1,3] . e1
    assert abs(y[0, 0, 0, 1] - 0.25) < tol
    assert abs(y[0, 1, 0, 0] - 2.0) < tol          # from W_1: row [2,3] . e1
    # second o-row: v = -0.5, vbar = 0.25 -> delta -0.75 -> [0.25-0.375, -0.5]
    assert abs(y[0, 1, 0, 1] - (-0.125)) < tol
    # step 2 moves row 0 by 0.5*(3-2) along e1 -> [2.5, 3]
    np.testing.assert_allclose(Wf[0, 0, 0], [2.5, 3.0], atol=tol, rtol=0)
    # the beta row stays 0 (its reads at k and q are both 0): gate stays 0.5
    np.testing.assert_allclose(Wf[0, 0, 6], [0.0, 0.0], atol=tol, rtol=0)


# ---------------------------------------------------------------- c2
@pytest.mark.parametrize("n_lr", [1, 4])
@pytest.mark.parametrize("softmax_input", [False, True])
def test_c2_zero_matrix_is_a_fixed_point(n_lr, softmax_input):
    """[REV] 2.5: with W0 = 0 both reads are 0, the update is 0, W stays 0."""
    d, H = 5, 2
    x = _rng(1).standard_normal((3, 9, H, d)).astype(np.float32)
    W0 = np.zeros((H, 3 * d + n_lr, d), np.float32)
    y, Wf = oracle.forward(x, W0, n_lr, softmax_input)
    assert not y.any() and not Wf.any()


# ---------------------------------------------------------------- c3
@pytest.mark.parametrize("d", [3, 8, 16])
def test_c3_readback_closed_form(d):
    """[REV] 2.3 derivation: after one update with fixed k=phi(k_t), q=phi(q_t),
    eta, the read-back at any address z is W'z = Wz + eta (k.z)(Wq - Wk); at the
    key itself W'k = Wk + eta ||k||^2 (Wq - Wk); and 1/d <= ||k||^2 <= 1."""
    r = _rng(d)
    m = 3 * d + 4
    W = r.standard_normal((m, d))
    k = sp_softmax(3 * r.standard_normal(d))
    q = sp_softmax(3 * r.standard_normal(d))
    # a different gate per row block, as in the four-learning-rate version
    etas = expit(r.standard_normal(4))
    gate = np.repeat(etas, [d, d, d, 4])
    W1 = oracle.delta_update(W, k, q, gate)
    diff = W @ q - W @ k
    n2 = float(k @ k)
    assert 1.0 / d - 1e-15 <= n2 <= 1.0 + 1e-15
    scale = np.abs(W).max()
    np.testing.assert_allclose(W1 @ k, W @ k + gate * n2 * diff, atol=1e-12 * scale, rtol=0)
    for _ in range(3):
        z = r.standard_normal(d)
        np.testing.assert_allclose(W1 @ z, W @ z + gate * float(k @ z) * diff,
                                   atol=1e-12 * scale * np.abs(z).sum(), rtol=0)


def test_c3_norm_bound_extremes():
    """||phi(k)||^2 reaches 1/d for equal logits and approaches 1 for one dominant logit."""
    d = 16
    k = sp_softmax(np.zeros(d))
    assert abs(k @ k - 1.0 / d) < 1e-15
    k = sp_softmax(np.r_[50.0, np.zeros(d - 1)])
    assert 1.0 - 1e-15 < k @ k <= 1.0


# ---------------------------------------------------------------- c4
def test_c4_one_rate_equals_four_rates_with_equal_gates():
    """Eq. (3) vs Eqs. (4)-(5): a 4-lr W0 whose four beta rows copy the 1-lr
    beta row has four equal learning rates at every step, so both versions
    produce the same y, and the 4-lr final beta rows are four copies."""
    r = _rng(4)
    d, H, B, T = 6, 3, 2, 20
    W1 = (r.standard_normal((H, 3 * d + 1, d)) / np.sqrt(d)).astype(np.float32)
    W4 = np.concatenate([W1[:, : 3 * d], np.repeat(W1[:, 3 * d:], 4, axis=1)], axis=1)
    x = r.standard_normal((B, T, H, d)).astype(np.float32)
    for smx in (False, True):
        y1, Wf1 = oracle.forward(x, W1, 1, smx)
        y4, Wf4 = oracle.forward(x, W4, 4, smx)
        np.testing.assert_array_equal(y1, y4)
        np.testing.assert_array_equal(Wf1[:, :, : 3 * d], Wf4[:, :, : 3 * d])
        for j in range(4):
            np.testing.assert_array_equal(Wf1[:, :, 3 * d], Wf4[:, :, 3 * d + j])


def test_c4_unequal_gates_do_differ():
    """The converse: distinct beta rows give distinct learning rates and change y."""
    r = _rng(5)
    d, T = 6, 12
    W4 = (r.standard_normal((1, 3 * d + 4, d)) / np.sqrt(d)).astype(np.float32)
    W4b = W4.copy()
    W4b[0, 3 * d + 0] += 1.0  # only beta^o differs
    x = r.standard_normal((1, T, 1, d)).astype(np.float32)
    y, _ = oracle.forward(x, W4, 4)
    yb, Wfb = oracle.forward(x, W4b, 4)
    assert np.array_equal(y[:, 0], yb[:, 0])       # step 0 reads W0 (beta unused yet)
    assert not np.allclose(y[:, 1:], yb[:, 1:])    # later outputs see the o-block gate


# ---------------------------------------------------------------- c5
def _brute(x, W0, n_lr, softmax_input):
    """Independent transcription: library softmax/sigmoid, whole-matrix algebra,
    and the update formed as an explicit m x d outer-product matrix G_t."""
    B, T, H, d = x.shape
    m = 3 * d + n_lr
    y = np.zeros((B, T, H, d))
    Wf = np.zeros((B, H, m, d))
    for b in range(B):
        for h in range(H):
            W = W0[h].astype(np.float64)
            for t in range(T):
                u = x[b, t, h].astype(np.float64)
                if softmax_input:
                    u = sp_softmax(u)
                o, k, q, beta = np.split(W @ u, [d, 2 * d, 3 * d])
                y[b, t, h] = o
                pk, pq = sp_softmax(k), sp_softmax(q)
                v, vbar = W @ pq, W @ pk
                if n_lr == 1:
                    g = np.full(m, expit(beta[0]))
                else:
                    g = np.repeat(expit(beta), [d, d, d, 4])
                G = np.outer(g * (v - vbar), pk)
                W = W + G
            Wf[b, h] = W
    return y, Wf


@pytest.mark.parametrize("d", [2, 3, 4])
@pytest.mark.parametrize("n_lr", [1, 4])
@pytest.mark.parametrize("softmax_input", [False, True])
def test_c5_brute_force_tiny(d, n_lr, softmax_input):
    r = _rng(100 * d + 10 * n_lr + softmax_input)
    B, T, H = 2, 16, 2
    x = (2 * r.standard_normal((B, T, H, d))).astype(np.float32)
    W0 = r.standard_normal((H, 3 * d + n_lr, d)).astype(np.float32)
    y, Wf = oracle.forward(x, W0, n_lr, softmax_input)
    yb, Wfb = _brute(x, W0, n_lr, softmax_input)
    assert _rel(y, yb) < 1e-13
    assert _rel(Wf, Wfb) < 1e-13


# ---------------------------------------------------------------- c6
@pytest.mark.parametrize("block", ["k", "q"])
def test_c6_softmax_shift_invariance(block):
    """Adding one row vector to every k-row (or q-row) of W0 shifts all logits
    of that block equally, so phi is unchanged; the update keeps the shift a
    common row vector, so y is unchanged at every step."""
    r = _rng(6 if block == "k" else 7)
    d, H, B, T, n_lr = 8, 2, 2, 50, 4
    # Dyadic values (multiples of 2^-12, |v| < 8) so that W0 + shift is exact in
    # float32: the shift then really is common to every row of the block.
    def dyadic(a):
        return (np.round(a * 4096.0) / 4096.0).astype(np.float32)

    W0 = dyadic(r.standard_normal((H, 3 * d + n_lr, d)) / np.sqrt(d))
    x = r.standard_normal((B, T, H, d)).astype(np.float32)
    lo = d if block == "k" else 2 * d
    W0s = W0.copy()
    W0s[:, lo:lo + d, :] += dyadic(r.standard_normal((H, 1, d)))
    assert np.array_equal(W0s[:, lo:lo + d] - W0[:, lo:lo + d],
                          np.broadcast_to(W0s[:, lo:lo + 1] - W0[:, lo:lo + 1], (H, d, d)))
    y, Wf = oracle.forward(x, W0, n_lr)
    ys, Wfs = oracle.forward(x, W0s, n_lr)
    assert _rel(ys, y) < 1e-11
    delta = Wfs[:, :, lo:lo + d, :] - Wf[:, :, lo:lo + d, :]
    spread = np.abs(delta - delta[:, :, :1, :]).max()
    assert spread < 1e-10 * np.abs(Wf).max()
    # the other blocks are untouched
    others = np.r_[0:lo, lo + d:3 * d + n_lr]
    assert _rel(Wfs[:, :, others], Wf[:, :, others]) < 1e-11


# ---------------------------------------------------------------- c7
@pytest.mark.parametrize("n_lr", [1, 4])
def test_c7_equal_k_and_q_rows_never_update(n_lr):
    """k-rows equal to q-rows give phi(q) = phi(k), so v = vbar and W stays W0:
    y_t = W0^o x_t, a plain matrix product."""
    r = _rng(8)
    d, H, B, T = 7, 3, 2, 11
    W0 = r.standard_normal((H, 3 * d + n_lr, d)).astype(np.float32)
    W0[:, 2 * d:3 * d] = W0[:, d:2 * d]
    x = r.standard_normal((B, T, H, d)).astype(np.float32)
    y, Wf = oracle.forward(x, W0, n_lr)
    ref = np.einsum("hod,bthd->btho", W0[:, :d].astype(np.float64), x.astype(np.float64))
    assert _rel(y, ref) < 1e-13
    np.testing.assert_array_equal(Wf, np.broadcast_to(W0, Wf.shape))


def test_c7_softmax_input_with_closed_gate():
    """softmax on x_t (the RL variant): beta rows of -50 give beta_t = -50 * sum(phi(x_t))
    = -50, gate ~ 2e-22, so W stays W0 to ~1e-20 and y_t = W0^o softmax(x_t)."""
    r = _rng(9)
    d, H, B, T = 8, 2, 3, 40
    W0 = r.standard_normal((H, 3 * d + 1, d)).astype(np.float32)
    W0[:, 3 * d:] = -50.0
    x = (2 * r.standard_normal((B, T, H, d))).astype(np.float32)
    y, _ = oracle.forward(x, W0, 1, softmax_input=True)
    xs = sp_softmax(x.astype(np.float64), axis=-1)
    ref = np.einsum("hod,bthd->btho", W0[:, :d].astype(np.float64), xs)
    assert _rel(y, ref) < 1e-12


# ---------------------------------------------------------------- layout
def test_heads_and_sequences_are_independent():
    """[REV] 2.4: each head runs its own SRWM on its own d coordinates, and W0 is
    shared by every sequence.  Slicing one (b, h) stream gives the same bits."""
    wl = inputs.workload("tiny").with_shape(B=3, H=4, T=9, d=5)
    x, W0 = inputs.make_inputs(wl)
    y, Wf = oracle.forward(x, W0, wl.n_lr)
    for b in range(3):
        for h in range(4):
            ys, Wfs = oracle.forward(x[b:b + 1, :, h:h + 1], W0[h:h + 1], wl.n_lr)
            np.testing.assert_array_equal(ys[0, :, 0], y[b, :, h])
            np.testing.assert_array_equal(Wfs[0, 0], Wf[b, h])


def test_per_sequence_initial_state_matches_shared():
    """Starting from per-sequence copies of W0 is the same as sharing W0."""
    wl = inputs.workload("tiny").with_shape(B=2, H=3, T=7, d=4)
    x, W0 = inputs.make_inputs(wl)
    y, Wf = oracle.forward(x, W0, wl.n_lr)
    W_seq = np.ascontiguousarray(np.broadcast_to(W0, (2,) + W0.shape))
    y2, Wf2 = oracle.forward(x, W_seq, wl.n_lr, per_sequence=True)
    np.testing.assert_array_equal(y, y2)
    np.testing.assert_array_equal(Wf, Wf2)


def test_zero_steps_returns_W0():
    W0 = _rng(3).standard_normal((2, 3 * 4 + 4, 4)).astype(np.float32)
    x = np.zeros((3, 0, 2, 4), np.float32)
    y, Wf = oracle.forward(x, W0, 4)
    assert y.shape == (3, 0, 2, 4)
    np.testing.assert_array_equal(Wf, np.broadcast_to(W0, Wf.shape))


# ---------------------------------------------------------------- c8
# Tolerances of the GPU parity bar: 1e-4 up to T = 1024, 1e-3 up to T = 8192.
def _bound(T):
    return 1e-4 if T <= 1024 else 1e-3


@pytest.mark.parametrize("name,pairs", [("tiny", None), ("fewshot", None), ("mid", (1, 2)),
                                        ("long", (1, 2)), ("rl", (2, 4))])
def test_c8_fp32_floor(name, pairs):
    """How far plain fp32 arithmetic (same operation order) drifts from the
    float64 oracle on each workload: the floor any fp32 implementation faces.
    Full T and d; the heavy workloads keep a few (b, h) streams."""
    wl = inputs.workload(name)
    if pairs is not None:
        wl = wl.with_shape(B=pairs[0], H=pairs[1])
    x, W0 = inputs.make_inputs(wl)
    y64, W64 = oracle.forward(x, W0, wl.n_lr, wl.softmax_input)
    y32, W32 = oracle.forward(x, W0, wl.n_lr, wl.softmax_input, precision="f32")
    ey, ew = _rel(y32, y64), _rel(W32, W64)
    print(f"fp32 floor {name}: y {ey:.3e}  W {ew:.3e}")
    assert ey < _bound(wl.T) and ew < _bound(wl.T)
