"""Python binding of libsrwm.so: argument marshalling only.

Every step of the recurrence runs in the library's sm_103a kernels; this
module checks tensor types, allocates outputs with torch when the caller does
not pass them, and forwards raw device pointers and the current CUDA stream.
If libsrwm.so is missing, every call raises: there is no fallback path.
"""
import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "libsrwm.so")
_LIB = None

# Status codes of include/srwm.h
SRWM_OK = 0
SRWM_ERR_SHAPE = 2
SRWM_ERR_TIMEOUT = 7

EXPORTS = ("srwm_forward", "srwm_forward_balanced", "srwm_forward_balanced_noalloc",
           "srwm_forward_workspace_bytes", "srwm_forward_from", "srwm_forward_host",
           "srwm_forward_host_workspace_bytes",
           "srwm_step", "srwm_backward", "srwm_backward_workspace_bytes",
           "srwm_layer_forward", "srwm_layer_workspace_bytes", "srwm_debug_set_layer_gemm", "srwm_status_string", "srwm_last_device_status", "srwm_set_wait_limit_ns",
           "srwm_debug_skip_x_chunk", "srwm_debug_set_segment_len", "srwm_debug_wrap_len",
           "srwm_debug_wrap_pieces", "srwm_debug_chunk_plan", "srwm_probe_fma")


class SrwmError(RuntimeError):
    """A libsrwm call returned a non-zero status."""

    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {srwm_status_string(status)} (status {status})")


def library_path() -> str:
    return _LIB_PATH


def _lib():
    global _LIB
    if _LIB is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"{_LIB_PATH} is not built. Build it with "
                "`python -m self_referential_weight_gb300.build` (needs nvcc).")
        lib = ctypes.CDLL(_LIB_PATH)
        P, I, LL = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong
        lib.srwm_forward.argtypes = [P, P, I, I, I, I, I, I, P, P, P]
        lib.srwm_forward.restype = I
        SZ = ctypes.c_size_t
        lib.srwm_forward_balanced.argtypes = [P, P, I, I, I, I, I, I, P, P, P, SZ, P]
        lib.srwm_forward_balanced.restype = I
        lib.srwm_forward_workspace_bytes.argtypes = [I, I]
        lib.srwm_forward_workspace_bytes.restype = SZ
        lib.srwm_forward_balanced_noalloc.argtypes = [P, P, I, I, I, I, I, I, P, P, P]
        lib.srwm_forward_balanced_noalloc.restype = I
        lib.srwm_debug_set_segment_len.argtypes = [I]
        lib.srwm_debug_set_segment_len.restype = I
        lib.srwm_debug_wrap_len.argtypes = [LL, I, LL, I]
        lib.srwm_debug_wrap_len.restype = LL
        lib.srwm_debug_wrap_pieces.argtypes = [LL, I, LL, LL, P, I]
        lib.srwm_debug_wrap_pieces.restype = I
        lib.srwm_debug_chunk_plan.argtypes = [I, I, I, P, I]
        lib.srwm_debug_chunk_plan.restype = I
        lib.srwm_forward_from.argtypes = [P, P, I, I, I, I, I, I, P, P, P]
        lib.srwm_forward_from.restype = I
        lib.srwm_forward_host.argtypes = [P, P, I, I, I, I, I, I, P, P, I, P, SZ, P]
        lib.srwm_forward_host.restype = I
        lib.srwm_forward_host_workspace_bytes.argtypes = [I, I, I, I, I, I]
        lib.srwm_forward_host_workspace_bytes.restype = SZ
        lib.srwm_step.argtypes = [P, P, I, I, I, I, I, P, P, P]
        lib.srwm_step.restype = I
        lib.srwm_backward.argtypes = [P, P, I, I, I, I, I, I, P, P, P, P, P, SZ, P]
        lib.srwm_backward.restype = I
        lib.srwm_backward_workspace_bytes.argtypes = [I, I, I, I, I]
        lib.srwm_backward_workspace_bytes.restype = SZ
        lib.srwm_layer_forward.argtypes = [P, I, I, I, I, I, I, P, P, P, P, P, P, P, I, P, P, P, P, P, SZ, P]
        lib.srwm_layer_forward.restype = I
        lib.srwm_layer_workspace_bytes.argtypes = [I, I, I, I, I, I]
        lib.srwm_layer_workspace_bytes.restype = SZ
        lib.srwm_debug_set_layer_gemm.argtypes = [I]
        lib.srwm_debug_set_layer_gemm.restype = I
        lib.srwm_status_string.argtypes = [I]
        lib.srwm_status_string.restype = ctypes.c_char_p
        lib.srwm_last_device_status.argtypes = [P]
        lib.srwm_last_device_status.restype = I
        lib.srwm_set_wait_limit_ns.argtypes = [LL]
        lib.srwm_set_wait_limit_ns.restype = I
        lib.srwm_debug_skip_x_chunk.argtypes = [I]
        lib.srwm_debug_skip_x_chunk.restype = I
        lib.srwm_probe_fma.argtypes = [I, I, I, I, P, P]
        lib.srwm_probe_fma.restype = I
        _LIB = lib
    return _LIB


def _stream_handle(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _dev(t, name, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous float32 CUDA tensor")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return ctypes.c_void_p(t.data_ptr() if t.numel() else 0)


def _check(rc, where):
    if rc != SRWM_OK:
        raise SrwmError(rc, where)


def srwm_status_string(status: int) -> str:
    return _lib().srwm_status_string(int(status)).decode()


def srwm_forward(x, W0, n_lr, softmax_input=False, y_out=None, W_final=None, stream=None):
    """T steps of the SRWM recurrence for every (sequence, head) stream.

    x [B,T,H,d] and W0 [H,m,d] (m = 3d + n_lr) are float32 CUDA tensors.
    Returns (y [B,T,H,d], W_final [B,H,m,d]); outputs are allocated when not given.
    """
    B, T, H, d = x.shape
    m = 3 * d + n_lr
    if y_out is None:
        y_out = torch.empty((B, T, H, d), dtype=torch.float32, device=x.device)
    if W_final is None:
        W_final = torch.empty((B, H, m, d), dtype=torch.float32, device=W0.device)
    px = _dev(x, "x")
    pw = _dev(W0, "W0", (H, m, d))
    py = _dev(y_out, "y_out", (B, T, H, d))
    pf = _dev(W_final, "W_final", (B, H, m, d))
    rc = _lib().srwm_forward(px, pw, B, T, H, d, int(n_lr), int(bool(softmax_input)), py, pf,
                             _stream_handle(stream))
    _check(rc, "srwm_forward")
    return y_out, W_final


def srwm_forward_workspace_bytes(B, H) -> int:
    return int(_lib().srwm_forward_workspace_bytes(int(B), int(H)))


def srwm_forward_balanced(x, W0, n_lr, softmax_input=False, y_out=None, W_final=None, workspace=None,
                          stream=None):
    """srwm_forward on the load-balanced segment schedule (same results).

    workspace: a CUDA tensor of at least srwm_forward_workspace_bytes(B, H)
    bytes (allocated here when not given)."""
    B, T, H, d = x.shape
    m = 3 * d + n_lr
    if y_out is None:
        y_out = torch.empty((B, T, H, d), dtype=torch.float32, device=x.device)
    if W_final is None:
        W_final = torch.empty((B, H, m, d), dtype=torch.float32, device=W0.device)
    nbytes = srwm_forward_workspace_bytes(B, H)
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=x.device)
    if not (workspace.is_cuda and workspace.is_contiguous()):
        raise ValueError("workspace must be a contiguous CUDA tensor")
    ws_bytes = workspace.numel() * workspace.element_size()
    rc = _lib().srwm_forward_balanced(_dev(x, "x"), _dev(W0, "W0", (H, m, d)), B, T, H, d, int(n_lr),
                                      int(bool(softmax_input)), _dev(y_out, "y_out", (B, T, H, d)),
                                      _dev(W_final, "W_final", (B, H, m, d)),
                                      ctypes.c_void_p(workspace.data_ptr()), ctypes.c_size_t(ws_bytes),
                                      _stream_handle(stream))
    _check(rc, "srwm_forward_balanced")
    return y_out, W_final


def srwm_forward_balanced_noalloc(x, W0, n_lr, softmax_input, y_out, W_final, stream=None):
    """srwm_forward_balanced with the library's own fixed scratch array instead
    of a workspace, for callers that cannot allocate device memory.  The
    outputs are the caller's (they must be given); B*H is at most 65536."""
    B, T, H, d = x.shape
    m = 3 * d + n_lr
    rc = _lib().srwm_forward_balanced_noalloc(_dev(x, "x"), _dev(W0, "W0", (H, m, d)), B, T, H, d, int(n_lr),
                                              int(bool(softmax_input)), _dev(y_out, "y_out", (B, T, H, d)),
                                              _dev(W_final, "W_final", (B, H, m, d)), _stream_handle(stream))
    _check(rc, "srwm_forward_balanced_noalloc")
    return y_out, W_final


def srwm_debug_wrap_len(n_streams: int, T: int, slots: int, tau: int) -> int:
    """Steps per warp slot of the wrap-around schedule (0: not used)."""
    return int(_lib().srwm_debug_wrap_len(int(n_streams), int(T), int(slots), int(tau)))


def srwm_debug_wrap_pieces(n_streams: int, T: int, wrap_len: int, slot: int):
    """The pieces of one slot under the wrap-around schedule, in run order:
    a list of (stream, segment, first step, steps)."""
    lib = _lib()
    n = lib.srwm_debug_wrap_pieces(int(n_streams), int(T), int(wrap_len), int(slot), None, 0)
    if n < 0:
        raise SrwmError(SRWM_ERR_SHAPE, "srwm_debug_wrap_pieces")
    buf = (ctypes.c_int * (4 * max(n, 1)))()
    lib.srwm_debug_wrap_pieces(int(n_streams), int(T), int(wrap_len), int(slot), buf, n)
    return [tuple(buf[4 * i:4 * i + 4]) for i in range(n)]


def srwm_debug_chunk_plan(T: int, d: int = 64, chunk_steps: int = 0):
    """The chunk lengths srwm_forward_host uses for T steps of width d."""
    lib = _lib()
    n = lib.srwm_debug_chunk_plan(int(T), int(d), int(chunk_steps), None, 0)
    if n < 0:
        raise SrwmError(SRWM_ERR_SHAPE, "srwm_debug_chunk_plan")
    buf = (ctypes.c_int * max(n, 1))()
    lib.srwm_debug_chunk_plan(int(T), int(d), int(chunk_steps), buf, n)
    return list(buf[:n])


def srwm_debug_set_segment_len(steps: int) -> None:
    _check(_lib().srwm_debug_set_segment_len(int(steps)), "srwm_debug_set_segment_len")


def srwm_forward_from(x, W_init, n_lr, softmax_input=False, y_out=None, W_final=None, stream=None):
    """T steps starting from per-sequence states W_init [B,H,m,d] (state carry).

    Returns (y [B,T,H,d], W_final [B,H,m,d]); W_final may be W_init itself."""
    B, T, H, d = x.shape
    m = 3 * d + n_lr
    if y_out is None:
        y_out = torch.empty((B, T, H, d), dtype=torch.float32, device=x.device)
    if W_final is None:
        W_final = torch.empty((B, H, m, d), dtype=torch.float32, device=W_init.device)
    rc = _lib().srwm_forward_from(_dev(x, "x"), _dev(W_init, "W_init", (B, H, m, d)), B, T, H, d,
                                  int(n_lr), int(bool(softmax_input)), _dev(y_out, "y_out", (B, T, H, d)),
                                  _dev(W_final, "W_final", (B, H, m, d)), _stream_handle(stream))
    _check(rc, "srwm_forward_from")
    return y_out, W_final


def _host(t, name, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != torch.float32 or t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous float32 CPU tensor (pinned for overlapped copies)")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return ctypes.c_void_p(t.data_ptr() if t.numel() else 0)


def srwm_forward_host_workspace_bytes(B, T, H, d, n_lr, chunk_steps=0) -> int:
    return int(_lib().srwm_forward_host_workspace_bytes(int(B), int(T), int(H), int(d), int(n_lr), int(chunk_steps)))


def srwm_forward_host(x, W0, n_lr, softmax_input=False, y_out=None, W_final=None, chunk_steps=0, workspace=None,
                      stream=None):
    """srwm_forward on host tensors (x [B,T,H,d], W0 [H,m,d], pinned for overlap):
    the copies to and from the device overlap the recurrence.  Returns
    (y, W_final) host tensors, written once `stream` has completed."""
    B, T, H, d = x.shape
    m = 3 * d + n_lr
    if y_out is None:
        y_out = torch.empty((B, T, H, d), dtype=torch.float32).pin_memory()
    if W_final is None:
        W_final = torch.empty((B, H, m, d), dtype=torch.float32).pin_memory()
    if workspace is None:
        need = srwm_forward_host_workspace_bytes(B, T, H, d, n_lr, chunk_steps)
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")
    rc = _lib().srwm_forward_host(_host(x, "x"), _host(W0, "W0", (H, m, d)), B, T, H, d, int(n_lr),
                                  int(bool(softmax_input)), _host(y_out, "y_out", (B, T, H, d)),
                                  _host(W_final, "W_final", (B, H, m, d)), int(chunk_steps),
                                  ctypes.c_void_p(workspace.data_ptr()),
                                  workspace.numel() * workspace.element_size(), _stream_handle(stream))
    _check(rc, "srwm_forward_host")
    return y_out, W_final


def srwm_step(x_t, W_in, n_lr, softmax_input=False, y_t=None, W_out=None, stream=None):
    """One step from per-sequence states: x_t [B,H,d], W_in [B,H,m,d] -> (y_t, W_out).

    W_out may be W_in itself (in-place update)."""
    B, H, d = x_t.shape
    m = 3 * d + n_lr
    if y_t is None:
        y_t = torch.empty((B, H, d), dtype=torch.float32, device=x_t.device)
    if W_out is None:
        W_out = torch.empty((B, H, m, d), dtype=torch.float32, device=W_in.device)
    rc = _lib().srwm_step(_dev(x_t, "x_t"), _dev(W_in, "W_in", (B, H, m, d)), B, H, d, int(n_lr),
                          int(bool(softmax_input)), _dev(y_t, "y_t", (B, H, d)),
                          _dev(W_out, "W_out", (B, H, m, d)), _stream_handle(stream))
    _check(rc, "srwm_step")
    return y_t, W_out


def srwm_backward_workspace_bytes(B, T, H, d, n_lr) -> int:
    return int(_lib().srwm_backward_workspace_bytes(int(B), int(T), int(H), int(d), int(n_lr)))


def srwm_backward(x, W0, n_lr, softmax_input, dy, dW_final=None, dx=None, dW0=None, workspace=None,
                  stream=None):
    """Gradients through srwm_forward(x, W0, ...): returns (dx [B,T,H,d], dW0 [H,m,d]).

    dy [B,T,H,d] = dL/dy; dW_final [B,H,m,d] = dL/dW_final or None (zero).
    The workspace is allocated when not given."""
    B, T, H, d = x.shape
    m = 3 * d + n_lr
    if dx is None:
        dx = torch.empty((B, T, H, d), dtype=torch.float32, device=x.device)
    if dW0 is None:
        dW0 = torch.empty((H, m, d), dtype=torch.float32, device=W0.device)
    need = srwm_backward_workspace_bytes(B, T, H, d, n_lr)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=x.device)
    if not isinstance(workspace, torch.Tensor) or not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    pf = _dev(dW_final, "dW_final", (B, H, m, d)) if dW_final is not None else ctypes.c_void_p(0)
    rc = _lib().srwm_backward(_dev(x, "x"), _dev(W0, "W0", (H, m, d)), B, T, H, d, int(n_lr),
                              int(bool(softmax_input)), _dev(dy, "dy", (B, T, H, d)), pf,
                              _dev(dx, "dx", (B, T, H, d)), _dev(dW0, "dW0", (H, m, d)),
                              ctypes.c_void_p(workspace.data_ptr()),
                              workspace.numel() * workspace.element_size(), _stream_handle(stream))
    _check(rc, "srwm_backward")
    return dx, dW0


def srwm_layer_workspace_bytes(B, T, H, d, n_lr, d_ff) -> int:
    return int(_lib().srwm_layer_workspace_bytes(int(B), int(T), int(H), int(d), int(n_lr), int(d_ff)))


def srwm_layer_forward(u, H, n_lr, softmax_input, ln1_gamma, ln1_beta, W0, ln2_gamma, ln2_beta, W1, b1, W2, b2,
                       out=None, W_final=None, workspace=None, stream=None):
    """One Recursive Self-Transformer layer: u [B,T,D] -> out [B,T,D] (D = H*d).

    Parameters as in include/srwm.h (W1 [d_ff,D], W2 [D,d_ff], PyTorch Linear
    layout).  W_final [B,H,m,d] receives the SRWM's final state when given."""
    B, T, D = u.shape
    d = D // H
    m = 3 * d + n_lr
    d_ff = W1.shape[0]
    if out is None:
        out = torch.empty((B, T, D), dtype=torch.float32, device=u.device)
    need = srwm_layer_workspace_bytes(B, T, H, d, n_lr, d_ff)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=u.device)
    if not isinstance(workspace, torch.Tensor) or not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    pwf = _dev(W_final, "W_final", (B, H, m, d)) if W_final is not None else ctypes.c_void_p(0)
    rc = _lib().srwm_layer_forward(
        _dev(u, "u"), B, T, H, d, int(n_lr), int(bool(softmax_input)), _dev(ln1_gamma, "ln1_gamma", (D,)),
        _dev(ln1_beta, "ln1_beta", (D,)), _dev(W0, "W0", (H, m, d)), _dev(ln2_gamma, "ln2_gamma", (D,)),
        _dev(ln2_beta, "ln2_beta", (D,)), _dev(W1, "W1", (d_ff, D)), _dev(b1, "b1", (d_ff,)), d_ff,
        _dev(W2, "W2", (D, d_ff)), _dev(b2, "b2", (D,)), _dev(out, "out", (B, T, D)), pwf,
        ctypes.c_void_p(workspace.data_ptr()), workspace.numel() * workspace.element_size(), _stream_handle(stream))
    _check(rc, "srwm_layer_forward")
    return out, W_final


def srwm_debug_set_layer_gemm(mode: int) -> None:
    """The layer's feed-forward products: 0 this library's tensor-core kernel
    (default), 1 cuBLASLt plain FP32, 2 cuBLASLt FP32 emulated on BF16 (the
    last two for comparison)."""
    _check(_lib().srwm_debug_set_layer_gemm(int(mode)), "srwm_debug_set_layer_gemm")


def srwm_last_device_status(stream=None) -> int:
    """Synchronise the stream; return (and clear) the kernels' status word."""
    return _lib().srwm_last_device_status(_stream_handle(stream))


def srwm_set_wait_limit_ns(limit_ns: int) -> None:
    _check(_lib().srwm_set_wait_limit_ns(int(limit_ns)), "srwm_set_wait_limit_ns")


def srwm_debug_skip_x_chunk(chunk: int) -> None:
    _check(_lib().srwm_debug_skip_x_chunk(int(chunk)), "srwm_debug_skip_x_chunk")


def srwm_probe_fma(blocks, threads, iters, packed, out, stream=None):
    rc = _lib().srwm_probe_fma(int(blocks), int(threads), int(iters), int(bool(packed)),
                               _dev(out, "out"), _stream_handle(stream))
    _check(rc, "srwm_probe_fma")
