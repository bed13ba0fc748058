"""Seeded synthetic inputs for the SRWM forward recurrence.

This module only draws numbers; it holds none of the recurrence's arithmetic.
The tests feed the same arrays to the CPU oracle and to the CUDA library, and
the benchmark uses it for its workloads.  It imports nothing else from the
package, so importing it never loads the CUDA library.

Generator (fixed, documented, platform independent):
  * SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
    generators", OOPSLA 2014) used in counter mode: output i of stream `key` is
    mix64(key + (i + 1) * 0x9E3779B97F4A7C15), with mix64 the SplitMix64
    finaliser.  The key of a stream is mix64(seed * 2**8 + tag) for a small tag
    per drawn quantity, so W0 does not depend on how many x values were drawn.
  * Uniform U = (output >> 11) * 2**-53 in [0, 1).
  * Normal pairs by Box-Muller: r = sqrt(-2 ln(1 - U_2j)),
    n_2j = r cos(2 pi U_2j+1), n_2j+1 = r sin(2 pi U_2j+1), rounded to float32.

Workloads (shapes, value distributions and structure of the pages' settings):
  tiny     B=1   T=64   H=1  d=16 n_lr=4 x ~ N(0,1)
  fewshot  B=128 T=26   H=16 d=16 n_lr=4 5-way 5-shot episodes: features N(0,1)
           in coordinates 0..250 of D=256, a one-hot label in the last five;
           25 support steps, then one query step with the label block empty
  mid      B=64  T=1024 H=8  d=64 n_lr=4 x ~ N(0,1)
  long     B=16  T=8192 H=8  d=64 n_lr=4 two tasks in sequence:
           x[b,t,:] = mu[b, seg(t)] + N(0, I_D), mu ~ N(0, I_D), seg switches at T/2
  rl       B=512 T=512  H=4  d=32 n_lr=1 x ~ N(0,1), softmax applied to x_t
W0 ~ N(0, 1/d) (standard deviation 1/sqrt(d)) in every workload.
"""
from __future__ import annotations

import dataclasses

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22  # normal pairs per chunk: bounds the temporaries to ~100 MB

# One tag per drawn quantity.
TAG_X, TAG_W0, TAG_MU, TAG_LABELS, TAG_DY, TAG_DWF, TAG_LAYER = 1, 2, 3, 4, 5, 6, 7


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    H: int
    d: int
    n_lr: int
    softmax_input: bool
    seed: int
    x_kind: str  # "normal" | "fewshot" | "two_task"

    @property
    def m(self) -> int:
        return 3 * self.d + self.n_lr

    @property
    def head_tokens(self) -> int:
        return self.B * self.T * self.H

    def with_shape(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny": Workload("tiny", 1, 64, 1, 16, 4, False, 0, "normal"),
    "fewshot": Workload("fewshot", 128, 26, 16, 16, 4, False, 1, "fewshot"),
    "mid": Workload("mid", 64, 1024, 8, 64, 4, False, 2, "normal"),
    "long": Workload("long", 16, 8192, 8, 64, 4, False, 3, "two_task"),
    "rl": Workload("rl", 512, 512, 4, 32, 1, True, 4, "normal"),
}


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, tag: int) -> np.uint64:
    with np.errstate(over="ignore"):
        return _mix64(np.array([(int(seed) << 8) + int(tag)], dtype=np.uint64))[0]


def uniforms(key: np.uint64, start: int, count: int) -> np.ndarray:
    """Outputs start .. start+count-1 of stream `key` as float64 in [0, 1)."""
    idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = _mix64(key + idx * _GAMMA)
    return (z >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)


def normals(key: np.uint64, count: int) -> np.ndarray:
    """`count` standard normal float32 values of stream `key` (Box-Muller)."""
    out = np.empty(count, dtype=np.float32)
    pairs = (count + 1) // 2
    for p0 in range(0, pairs, _CHUNK):
        p1 = min(pairs, p0 + _CHUNK)
        u = uniforms(key, 2 * p0, 2 * (p1 - p0))
        r = np.sqrt(-2.0 * np.log1p(-u[0::2]))
        ang = (2.0 * np.pi) * u[1::2]
        n = np.empty(2 * (p1 - p0), dtype=np.float64)
        n[0::2] = r * np.cos(ang)
        n[1::2] = r * np.sin(ang)
        lo = 2 * p0
        hi = min(count, 2 * p1)
        out[lo:hi] = n[: hi - lo]
    return out


def make_W0(H: int, d: int, n_lr: int, seed: int) -> np.ndarray:
    """W0 [H, m, d] float32 ~ N(0, 1/d)."""
    m = 3 * d + n_lr
    w = normals(stream_key(seed, TAG_W0), H * m * d).reshape(H, m, d)
    return (w * np.float32(1.0 / np.sqrt(d))).astype(np.float32)


def make_x(wl: Workload) -> np.ndarray:
    """x [B, T, H, d] float32 with the workload's structure."""
    B, T, H, d = wl.B, wl.T, wl.H, wl.d
    D = H * d
    x = normals(stream_key(wl.seed, TAG_X), B * T * D).reshape(B, T, D)
    if wl.x_kind == "two_task":
        mu = normals(stream_key(wl.seed, TAG_MU), B * 2 * D).reshape(B, 2, D)
        half = T // 2
        x[:, :half, :] += mu[:, 0:1, :]
        x[:, half:, :] += mu[:, 1:2, :]
    elif wl.x_kind == "fewshot":
        n_way = 5
        if D < n_way:
            raise ValueError("few-shot episodes need at least 5 input coordinates")
        support = T - 1
        x[:, :, D - n_way:] = 0.0
        for b in range(B):
            # A seeded order of the support labels (k copies of each class).
            u = uniforms(stream_key(wl.seed, TAG_LABELS), b * max(support, 1), support)
            labels = (np.arange(support) % n_way)[np.argsort(u, kind="stable")]
            x[b, np.arange(support), D - n_way + labels] = 1.0
        # The last step is the query: features only, label block left empty.
    elif wl.x_kind != "normal":
        raise ValueError(f"unknown x_kind {wl.x_kind!r}")
    return np.ascontiguousarray(x.reshape(B, T, H, d))


def make_inputs(wl: Workload):
    """(x [B,T,H,d], W0 [H,m,d]) float32 for a workload."""
    return make_x(wl), make_W0(wl.H, wl.d, wl.n_lr, wl.seed)


def make_cotangents(wl: Workload, with_dW_final: bool = True):
    """Output cotangents of a loss for a backward pass: (dy [B,T,H,d],
    dW_final [B,H,m,d] or None), float32 ~ N(0, 1)."""
    B, T, H, d = wl.B, wl.T, wl.H, wl.d
    m = 3 * d + wl.n_lr
    dy = normals(stream_key(wl.seed, TAG_DY), B * T * H * d).reshape(B, T, H, d)
    dWf = None
    if with_dW_final:
        dWf = normals(stream_key(wl.seed, TAG_DWF), B * H * m * d).reshape(B, H, m, d)
    return dy, dWf


def make_layer_params(H: int, d: int, n_lr: int, d_ff: int, seed: int) -> dict:
    """Seeded float32 parameters of one Recursive Self-Transformer layer:
    layer-norm scales ~ 1 + N(0, 0.1^2) and shifts ~ N(0, 0.1^2), W0 ~ N(0, 1/d)
    per head, feed-forward weights ~ N(0, 1/fan_in) and biases ~ N(0, 0.1^2)."""
    D = H * d
    key = stream_key(seed, TAG_LAYER)
    sizes = [("ln1_gamma", (D,)), ("ln1_beta", (D,)), ("ln2_gamma", (D,)), ("ln2_beta", (D,)),
             ("W1", (d_ff, D)), ("b1", (d_ff,)), ("W2", (D, d_ff)), ("b2", (D,))]
    total = sum(int(np.prod(s)) for _, s in sizes)
    z = normals(key, total)
    out, off = {}, 0
    for name, shape in sizes:
        n = int(np.prod(shape))
        v = z[off:off + n].reshape(shape).astype(np.float64)
        off += n
        if name.endswith("gamma"):
            v = 1.0 + 0.1 * v
        elif name in ("W1", "W2"):
            v = v / np.sqrt(shape[1])
        else:
            v = 0.1 * v
        out[name] = np.ascontiguousarray(v.astype(np.float32))
    out["W0"] = make_W0(H, d, n_lr, seed)
    return out


def make_layer_input(B: int, T: int, D: int, seed: int) -> np.ndarray:
    """Layer input tokens u [B, T, D] float32 ~ N(0, 1)."""
    return normals(stream_key(seed, TAG_X), B * T * D).reshape(B, T, D)


def workload(name: str, **overrides) -> Workload:
    wl = WORKLOADS[name]
    return wl.with_shape(**overrides) if overrides else wl
