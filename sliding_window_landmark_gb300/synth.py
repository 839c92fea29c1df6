"""Seeded synthetic inputs for sealed O(1) layers.

Counter-based, so any element of any tensor is reproducible from
(seed, layer, tensor, index) alone, whatever slice of a prompt is asked for:
SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014; the finaliser as published by Vigna) feeds the
Box-Muller transform (Box and Muller, 1958) in double, and the result is
rounded to f32. This module holds none of the attention method's arithmetic;
both the CUDA path's tests and the oracle take their inputs from it.

Also here: the integer "jit" pattern the pages' own batch-vs-serial tests use
(``jit(a, b) = ((37a + 13b + 3) mod 83) / 83 - 0.5``), and the workload shapes.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# Tensor ids of a layer's inputs.
Q, K, V, GATE, SINK_K, SINK_V, K_TILDE, Q_TILDE, MU = range(1, 10)


def _mix(z: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        z = z + _GAMMA
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def _stream(seed: int, layer: int, tensor: int) -> np.uint64:
    s = _mix(np.array([seed], dtype=np.uint64))
    s = _mix(s ^ np.uint64(layer))
    s = _mix(s ^ np.uint64(tensor))
    return s[0]


def normal(seed: int, layer: int, tensor: int, shape, offset: int = 0, absolute: bool = False) -> np.ndarray:
    """N(0,1) entries (f32) of ``shape``, element i being stream index offset + i."""
    n = int(np.prod(shape))
    base = _stream(seed, layer, tensor)
    idx = np.arange(offset, offset + n, dtype=np.uint64)
    with np.errstate(over="ignore"):
        c = base + idx * np.uint64(2)
        z1 = _mix(c)
        z2 = _mix(c + np.uint64(1))
    u1 = ((z1 >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)
    u2 = (z2 >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)
    x = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
    if absolute:
        x = np.abs(x)
    return x.astype(np.float32).reshape(shape)


def jit(a, b) -> np.ndarray:
    """The pages' deterministic test pattern, as f32."""
    a = np.asarray(a, dtype=np.int64)
    return (((a * 37 + b * 13 + 3) % 83).astype(np.float32) / np.float32(83.0) - np.float32(0.5)).astype(np.float32)


@dataclass
class Shape:
    """One sealed layer's shape (``window`` = ring stride = widest group window)."""
    groups: int
    heads_per_group: int
    d: int
    dv: int
    sinks: int
    window: int
    landmarks: int
    rope_base: float = 1e6
    group_windows: tuple | None = None

    @property
    def nh(self) -> int:
        return self.groups * self.heads_per_group


@dataclass
class LayerInputs:
    """Everything one layer needs: constants of the sealed state and the rows."""
    shape: Shape
    sink_k: np.ndarray
    sink_v: np.ndarray
    k_tilde: np.ndarray
    q_tilde: np.ndarray
    mu: np.ndarray
    extra: dict = field(default_factory=dict)


def layer_constants(shape: Shape, seed: int, layer: int = 0, mu_abs: bool = False) -> LayerInputs:
    s = shape
    return LayerInputs(
        shape=s,
        sink_k=normal(seed, layer, SINK_K, (s.groups, s.sinks, s.d)),
        sink_v=normal(seed, layer, SINK_V, (s.groups, s.sinks, s.dv)),
        k_tilde=normal(seed, layer, K_TILDE, (s.groups, s.landmarks, s.d)),
        q_tilde=normal(seed, layer, Q_TILDE, (s.groups, s.heads_per_group, s.landmarks, s.d)),
        mu=normal(seed, layer, MU, (s.nh, s.landmarks, s.landmarks), absolute=mu_abs),
    )


def layer_rows(shape: Shape, seed: int, row0: int, rows: int, layer: int = 0, gate: bool = True):
    """q, k, v, gate of prompt rows [row0, row0 + rows): the same values whatever
    the split of a prompt into calls."""
    s = shape
    q = normal(seed, layer, Q, (rows, s.nh, s.d), offset=row0 * s.nh * s.d)
    k = normal(seed, layer, K, (rows, s.groups, s.d), offset=row0 * s.groups * s.d)
    v = normal(seed, layer, V, (rows, s.groups, s.dv), offset=row0 * s.groups * s.dv)
    g = normal(seed, layer, GATE, (rows, s.nh, s.dv), offset=row0 * s.nh * s.dv) if gate else None
    return q, k, v, g


# The workloads: a tiny case the oracle finishes instantly; a single layer of
# Qwen3.5-0.8B shape (2 KV groups x 4 query heads, d = dv = 256); its decode
# path; a long prompt with per-group windows; a stack of 24 layers.
TINY = Shape(groups=1, heads_per_group=2, d=64, dv=64, sinks=4, window=16, landmarks=4)
QWEN_LAYER = Shape(groups=2, heads_per_group=4, d=256, dv=256, sinks=4, window=2048, landmarks=32)
QWEN_LONG = Shape(groups=2, heads_per_group=4, d=256, dv=256, sinks=4, window=2048, landmarks=32,
                  group_windows=(1024, 2048))
STACK_LAYER = Shape(groups=4, heads_per_group=4, d=128, dv=128, sinks=4, window=1024, landmarks=64)
