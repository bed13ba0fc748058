"""Gradient oracle of the SRWM recurrence (test infrastructure only).

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may use
it.  The forward recurrence is written a second time here in plain PyTorch
float64 CPU operations, step by step in the notation of "Metalearning
Continual Learning Algorithms", section 2.3 (Eqs. (1)-(3); four learning
rates, Eqs. (4)-(5)), and differentiated by autograd (a library routine).  It
is pinned in tests/test_oracle_grad_pins.py against the C oracle's forward,
finite differences, a closed form and the one-rate / four-rate equivalence.

The loss whose gradients are returned is L = <dy, y> + <dW_final, W_final>,
so dx = dL/dx and dW0 = dL/dW0 for given output cotangents dy, dW_final.
"""
import numpy as np
import torch


def _gates(beta, n_lr, d):
    """sigma(beta) of the block that owns each row: [.., m]."""
    g = torch.sigmoid(beta)
    if n_lr == 1:
        return g[..., :1].expand(*g.shape[:-1], 3 * d + 1)
    return torch.cat([g[..., 0:1].expand(*g.shape[:-1], d), g[..., 1:2].expand(*g.shape[:-1], d),
                      g[..., 2:3].expand(*g.shape[:-1], d), g[..., 3:4].expand(*g.shape[:-1], 4)], dim=-1)


def forward_torch(x, W_init, n_lr, softmax_input=False, per_sequence=False):
    """x [B,T,H,d] and W_init [H,m,d] (or [B,H,m,d]) float64 tensors -> (y, W_final)."""
    B, T, H, d = x.shape
    W = W_init.expand(B, H, *W_init.shape[-2:]) if not per_sequence else W_init
    ys = []
    for t in range(T):
        u = x[:, t]                                   # [B,H,d]
        if softmax_input:
            u = torch.softmax(u, dim=-1)
        z = torch.einsum("bhmd,bhd->bhm", W, u)       # Eq. (1)
        ys.append(z[..., :d])                         # output from W_{t-1}
        k, q, beta = z[..., d:2 * d], z[..., 2 * d:3 * d], z[..., 3 * d:]
        pk, pq = torch.softmax(k, dim=-1), torch.softmax(q, dim=-1)
        v = torch.einsum("bhmd,bhd->bhm", W, pq)      # Eq. (2)
        vbar = torch.einsum("bhmd,bhd->bhm", W, pk)
        g = _gates(beta, n_lr, d)
        W = W + (g * (v - vbar)).unsqueeze(-1) * pk.unsqueeze(-2)   # Eq. (3) / (5)
    return torch.stack(ys, dim=1), W


def grads(x, W0, n_lr, softmax_input, dy, dW_final=None):
    """Gradients of L = <dy, y> + <dW_final, W_final> (numpy in, numpy out).

    x [B,T,H,d], W0 [H,m,d], dy [B,T,H,d], dW_final [B,H,m,d] or None.
    Returns (dx [B,T,H,d], dW0 [H,m,d]) in float64.
    """
    xt = torch.tensor(np.asarray(x, np.float64), requires_grad=True)
    Wt = torch.tensor(np.asarray(W0, np.float64), requires_grad=True)
    y, Wf = forward_torch(xt, Wt, n_lr, softmax_input)
    loss = (y * torch.tensor(np.asarray(dy, np.float64))).sum()
    if dW_final is not None:
        loss = loss + (Wf * torch.tensor(np.asarray(dW_final, np.float64))).sum()
    loss.backward()
    return xt.grad.numpy(), Wt.grad.numpy()
