"""ctypes front end of the C oracle (oracle/srwm_oracle.c).

TEST INFRASTRUCTURE: only tests/, __graft_entry__.smoke() and bench.py's
CPU-baseline leg may call it.  It marshals numpy arrays; every step of the
recurrence runs in the C code, which follows "Metalearning Continual Learning
Algorithms", section 2.3, Eqs. (1)-(5).
"""
import ctypes
import os

import numpy as np

from . import build as _build

_LIB = None


def lib_path() -> str:
    return _build.LIB


def _lib():
    global _LIB
    if _LIB is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I = ctypes.c_int
        for name in ("srwm_oracle_forward_f64", "srwm_oracle_forward_f32"):
            fn = getattr(lib, name)
            fn.argtypes = [P, P, I, I, I, I, I, I, I, P, P, I]
            fn.restype = I
        lib.srwm_oracle_delta_update.argtypes = [P, I, I, P, P, P]
        lib.srwm_oracle_delta_update.restype = I
        _LIB = lib
    return _LIB


def _ptr(a):
    return ctypes.c_void_p(a.ctypes.data) if a is not None and a.size else None


def forward(x, W_init, n_lr, softmax_input=False, *, per_sequence=False, precision="f64",
            n_threads=None):
    """Run the SRWM recurrence on the CPU.

    x       : [B, T, H, d] float32
    W_init  : [H, m, d] float32 shared by every sequence, or [B, H, m, d] float32
              when per_sequence is True; m = 3d + n_lr
    returns : (y [B, T, H, d], W_final [B, H, m, d]) in float64 (precision "f64")
              or float32 (precision "f32", the fp32-floor measurement mode)
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    W_init = np.ascontiguousarray(W_init, dtype=np.float32)
    if x.ndim != 4:
        raise ValueError("x must be [B, T, H, d]")
    B, T, H, d = x.shape
    m = 3 * d + n_lr
    want = (B, H, m, d) if per_sequence else (H, m, d)
    if W_init.shape != want:
        raise ValueError(f"W_init has shape {W_init.shape}, expected {want}")
    dt = np.float64 if precision == "f64" else np.float32
    y = np.empty((B, T, H, d), dtype=dt)
    W_final = np.empty((B, H, m, d), dtype=dt)
    if n_threads is None:
        n_threads = os.cpu_count() or 1
    fn = _lib().srwm_oracle_forward_f64 if precision == "f64" else _lib().srwm_oracle_forward_f32
    rc = fn(_ptr(x), _ptr(W_init), int(per_sequence), B, T, H, d, n_lr, int(bool(softmax_input)),
            _ptr(y), _ptr(W_final), int(n_threads))
    if rc != 0:
        raise RuntimeError(f"oracle forward failed with code {rc}")
    return y, W_final


def delta_update(W, phi_k, phi_q, gate_of_row):
    """One delta-rule update with given addresses (Eqs. (2)-(3)), in float64.

    W [m, d], phi_k [d], phi_q [d], gate_of_row [m]; returns the updated copy of W.
    """
    W = np.array(W, dtype=np.float64, order="C", copy=True)
    m, d = W.shape
    phi_k = np.ascontiguousarray(phi_k, dtype=np.float64)
    phi_q = np.ascontiguousarray(phi_q, dtype=np.float64)
    g = np.ascontiguousarray(gate_of_row, dtype=np.float64)
    if phi_k.shape != (d,) or phi_q.shape != (d,) or g.shape != (m,):
        raise ValueError("shape mismatch")
    rc = _lib().srwm_oracle_delta_update(_ptr(W), m, d, _ptr(phi_k), _ptr(phi_q), _ptr(g))
    if rc != 0:
        raise RuntimeError(f"oracle delta_update failed with code {rc}")
    return W
