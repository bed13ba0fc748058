"""Host-only checks of the C ABI (no GPU needed): the library builds, exports
every entry point declared in include/srwm.h, and rejects bad arguments before
touching CUDA."""
import ctypes
import os
import re

import pytest

from self_referential_weight_gb300 import build as lib_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "srwm.h")


@pytest.fixture(scope="module")
def lib():
    path = lib_build.build()
    L = ctypes.CDLL(path)
    P, I = ctypes.c_void_p, ctypes.c_int
    L.srwm_forward.argtypes = [P, P, I, I, I, I, I, I, P, P, P]
    L.srwm_step.argtypes = [P, P, I, I, I, I, I, P, P, P]
    L.srwm_status_string.restype = ctypes.c_char_p
    return L


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:int|size_t|long long|const char\*)\s+(srwm_\w+)\s*\(", text, re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("srwm_forward", "srwm_step", "srwm_status_string", "srwm_last_device_status"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_binding_lists_the_same_exports():
    from self_referential_weight_gb300 import binding
    assert sorted(binding.EXPORTS) == declared_functions()


A = 0x100000  # fake, 16-byte aligned "device" addresses: never dereferenced


def fwd(lib, x=A, W0=A + 0x1000000, B=2, T=3, H=2, d=16, n_lr=4, smx=0, y=A + 0x2000000,
        Wf=A + 0x3000000):
    return lib.srwm_forward(x, W0, B, T, H, d, n_lr, smx, y, Wf, None)


def test_null_pointers(lib):
    assert fwd(lib, x=None) == 1
    assert fwd(lib, W0=None) == 1
    assert fwd(lib, y=None) == 1
    assert fwd(lib, Wf=None) == 1
    assert lib.srwm_step(None, A, 1, 1, 16, 4, 0, A, A, None) == 1


def test_bad_shapes(lib):
    assert fwd(lib, B=0) == 2
    assert fwd(lib, H=-1) == 2
    assert fwd(lib, T=-1) == 2
    assert fwd(lib, d=0) == 2
    assert fwd(lib, B=1 << 20, H=1 << 12) == 2  # more than 2^31 streams


def test_unsupported(lib):
    assert fwd(lib, d=48) == 3
    assert fwd(lib, d=128) == 3
    assert fwd(lib, n_lr=2) == 3
    assert fwd(lib, smx=2) == 3


def test_alignment(lib):
    assert fwd(lib, x=A + 4) == 4
    assert fwd(lib, Wf=A + 0x3000008) == 4


def test_aliasing(lib):
    # y overlapping x, W_final overlapping y
    assert fwd(lib, y=A) == 5
    assert fwd(lib, Wf=A + 0x2000000 + 64) == 5
    # step: exact in-place W is allowed past the alias check, partial overlap is not
    assert lib.srwm_step(A, A + 0x1000000, 1, 1, 16, 4, 0, A + 0x2000000, A + 0x1000000 + 16, None) == 5


def test_status_strings(lib):
    for code in range(9):
        s = lib.srwm_status_string(code).decode()
        assert s.startswith("SRWM")
    assert "unknown" in lib.srwm_status_string(99).decode()


def test_oracle_library_is_separate():
    """The oracle is its own library; the CUDA library exports none of its symbols."""
    import oracle
    from oracle import build as ob
    ob.build()
    names = set(re.findall(r"\b(srwm_oracle_\w+)", open(os.path.join(ROOT, "oracle", "srwm_oracle.c")).read()))
    lib = ctypes.CDLL(lib_build.LIB)
    for n in names:
        assert not hasattr(lib, n)
    assert oracle.lib_path() != lib_build.LIB


def test_forward_from_validation(lib):
    P, I = ctypes.c_void_p, ctypes.c_int
    lib.srwm_forward_from.argtypes = [P, P, I, I, I, I, I, I, P, P, P]
    ok = dict(x=A, W=A + 0x1000000, y=A + 0x2000000, Wf=A + 0x3000000)

    def call(**kw):
        a = dict(ok, **kw)
        return lib.srwm_forward_from(a["x"], a["W"], 2, 3, 2, 16, 4, 0, a["y"], a["Wf"], None)

    assert call(W=None) == 1
    assert call(x=A + 4) == 4
    assert call(Wf=A + 0x1000000 + 16) == 5      # partial overlap of W_final with W_init
    assert lib.srwm_forward_from(A, A + 0x1000000, 2, 3, 2, 48, 4, 0, A + 0x2000000, A + 0x3000000, None) == 3


def test_forward_balanced_validation(lib):
    P, I, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lib.srwm_forward_balanced.argtypes = [P, P, I, I, I, I, I, I, P, P, P, SZ, P]
    lib.srwm_forward_workspace_bytes.argtypes = [I, I]
    lib.srwm_forward_workspace_bytes.restype = SZ
    need = lib.srwm_forward_workspace_bytes(2, 2)
    assert need >= 2 * 2 * 4 and need % 256 == 0
    assert lib.srwm_forward_workspace_bytes(0, 2) == 0
    ws = A + 0x4000000

    def call(ws=ws, nbytes=need, **kw):
        return lib.srwm_forward_balanced(A, A + 0x1000000, 2, 3, 2, 16, 4, 0, A + 0x2000000,
                                         A + 0x3000000, ws, nbytes, None)

    assert call(ws=None) == 1
    assert call(nbytes=8) == 2
    assert call(ws=ws + 4) == 4
    assert call(ws=A + 0x2000000 + 64) == 5      # workspace inside y_out


def test_debug_segment_len_rejects_bad_values(lib):
    assert lib.srwm_debug_set_segment_len(33) == 2
    assert lib.srwm_debug_set_segment_len(-32) == 2
    assert lib.srwm_debug_set_segment_len(0) == 0


def test_backward_workspace_bytes(lib):
    L = lib
    SZ, I = ctypes.c_size_t, ctypes.c_int
    L.srwm_backward_workspace_bytes.argtypes = [I, I, I, I, I]
    L.srwm_backward_workspace_bytes.restype = SZ
    # regions, each rounded up to 256 bytes: dL/dW0 per stream and W_T
    # (B*H*m*d floats each), the forward's y (B*T*H*d), the per-step records
    # (B*H*T records of ceil4(5d + 4 + n_lr) floats), the counters (B*H ints)
    def expect(B, T, H, d, n_lr):
        a = lambda n: (n + 255) // 256 * 256
        m = 3 * d + n_lr
        rec = (5 * d + 4 + n_lr + 3) // 4 * 4
        return 2 * a(4 * B * H * m * d) + a(4 * B * T * H * d) + a(4 * B * H * T * rec) + a(4 * B * H)
    for B, T, H, d, n_lr in [(2, 75, 3, 16, 4), (1, 32, 1, 64, 1), (5, 1, 2, 32, 4), (64, 1024, 8, 64, 4)]:
        assert L.srwm_backward_workspace_bytes(B, T, H, d, n_lr) == expect(B, T, H, d, n_lr)
    assert L.srwm_backward_workspace_bytes(2, 0, 3, 16, 4) == expect(2, 0, 3, 16, 4)
    assert L.srwm_backward_workspace_bytes(2, 5, 3, 48, 4) == 0
    assert L.srwm_backward_workspace_bytes(2, 5, 3, 16, 2) == 0
    assert L.srwm_backward_workspace_bytes(0, 5, 3, 16, 4) == 0


def test_backward_validation(lib):
    P, I, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lib.srwm_backward.argtypes = [P, P, I, I, I, I, I, I, P, P, P, P, P, SZ, P]
    big = 1 << 40

    def bwd(x=A, W0=A + 0x1000000, B=2, T=3, H=2, d=16, n_lr=4, smx=0, dy=A + 0x2000000, dWf=None,
            dx=A + 0x3000000, dW0=A + 0x4000000, ws=A + 0x5000000, ws_bytes=big):
        return lib.srwm_backward(x, W0, B, T, H, d, n_lr, smx, dy, dWf, dx, dW0, ws, ws_bytes, None)

    assert bwd(x=None) == 1 and bwd(dy=None) == 1 and bwd(dx=None) == 1
    assert bwd(W0=None) == 1 and bwd(dW0=None) == 1 and bwd(ws=None) == 1
    assert bwd(B=0) == 2 and bwd(T=-1) == 2
    assert bwd(d=8) == 3 and bwd(n_lr=2) == 3 and bwd(smx=2) == 3
    assert bwd(ws_bytes=1024) == 2          # too small for these sizes
    assert bwd(dx=A + 0x3000004) == 4       # misaligned
    assert bwd(dx=A + 0x2000000) == 5       # dx on top of dy
    assert bwd(ws=A) == 5                   # workspace over x


def test_layer_workspace_and_validation(lib):
    P, I, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lib.srwm_layer_workspace_bytes.argtypes = [I, I, I, I, I, I]
    lib.srwm_layer_workspace_bytes.restype = SZ
    lib.srwm_layer_forward.argtypes = [P, I, I, I, I, I, I, P, P, P, P, P, P, P, I, P, P, P, P, P, SZ, P]
    ws = lib.srwm_layer_workspace_bytes
    assert ws(2, 10, 2, 16, 4, 128) > 32 << 20          # activations plus the GEMM scratch
    assert ws(2, 10, 2, 16, 4, 130) == 0                # d_ff % 4 != 0
    assert ws(2, 10, 32, 64, 4, 128) == 0               # D = 2048 > 1024
    assert ws(2, 10, 2, 48, 4, 128) == 0                # d unsupported
    grow = ws(2, 20, 2, 16, 4, 128) - ws(2, 10, 2, 16, 4, 128)
    assert grow >= 2 * 10 * (2 * 2 * 16 + 128) * 4      # a, y and the hidden layer scale with B*T

    base = 0x100000
    args = dict(u=base, B=2, T=3, H=2, d=16, n_lr=4, smx=0, g1=base + 0x10000, be1=base + 0x20000,
                W0=base + 0x30000, g2=base + 0x40000, be2=base + 0x50000, W1=base + 0x60000, b1=base + 0x70000,
                d_ff=64, W2=base + 0x80000, b2=base + 0x90000, out=base + 0xA0000, Wf=None, ws=base + 0x1000000,
                ws_bytes=1 << 30)

    def call(**kw):
        a = dict(args, **kw)
        return lib.srwm_layer_forward(a["u"], a["B"], a["T"], a["H"], a["d"], a["n_lr"], a["smx"], a["g1"], a["be1"],
                                      a["W0"], a["g2"], a["be2"], a["W1"], a["b1"], a["d_ff"], a["W2"], a["b2"],
                                      a["out"], a["Wf"], a["ws"], a["ws_bytes"], None)

    assert call(u=None) == 1 and call(W1=None) == 1 and call(ws=None) == 1
    assert call(B=0) == 2 and call(T=-1) == 2
    assert call(d=48) == 3 and call(d_ff=66) == 3 and call(H=32, d=64) == 3
    assert call(ws_bytes=1024) == 2
    assert call(out=base + 0xA0004) == 4
    assert call(out=base) == 5                          # out over u


def test_layer_gemm_mode_is_checked(lib):
    lib.srwm_debug_set_layer_gemm.argtypes = [ctypes.c_int]
    lib.srwm_debug_set_layer_gemm.restype = ctypes.c_int
    assert lib.srwm_debug_set_layer_gemm(3) == 3    # SRWM_ERR_UNSUPPORTED
    assert lib.srwm_debug_set_layer_gemm(-1) == 3
    assert lib.srwm_debug_set_layer_gemm(0) == 0


def test_layer_hidden_width_must_be_a_multiple_of_8(lib):
    lib.srwm_layer_workspace_bytes.argtypes = [ctypes.c_int] * 6
    lib.srwm_layer_workspace_bytes.restype = ctypes.c_size_t
    assert lib.srwm_layer_workspace_bytes(2, 8, 2, 16, 4, 64) > 0
    assert lib.srwm_layer_workspace_bytes(2, 8, 2, 16, 4, 12) == 0
