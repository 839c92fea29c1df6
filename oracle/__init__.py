"""Serial CPU oracle of a sealed O(1) attention layer (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package. It is a plain, slow, double-precision
restatement of the method, one row at a time, written in C (``o1_oracle.c``)
and wrapped here with ctypes and numpy. It shares nothing with the CUDA
library: no code, header, table or constant.

The method follows "cortiq-engine 0.8.51 src/gpu_wgpu/o1_batch.rs" (module
doc and kernels o1b_far_e / o1b_attend / o1b_far_commit / o1b_ring_commit /
o1b_meta), with the rotation of "cortiq-engine 0.8.77 src/gpu_wgpu/dory.rs"
(dory_prep and the rotary table of ``run``) and its output gate (dory_gate1).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "o1_oracle.c")
_LIB = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain C, -O2, no vector intrinsics)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
             "-ffp-contract=off", _SRC, "-o", tmp, "-lm", "-lpthread"])
        os.replace(tmp, _LIB)
    return _LIB


class _Geom(ctypes.Structure):
    _fields_ = [("groups", ctypes.c_int32), ("hpg", ctypes.c_int32),
                ("d", ctypes.c_int32), ("dv", ctypes.c_int32),
                ("sinks", ctypes.c_int32), ("window", ctypes.c_int32),
                ("landmarks", ctypes.c_int32), ("rect", ctypes.c_int32),
                ("scale", ctypes.c_float), ("rope_base", ctypes.c_float)]


_P = ctypes.c_void_p


class _State(ctypes.Structure):
    _fields_ = [("meta", _P), ("pos", _P), ("ring_k", _P), ("ring_v", _P),
                ("sink_k", _P), ("sink_v", _P), ("kt", _P), ("qt", _P), ("mu", _P),
                ("M", _P), ("Z", _P), ("T", _P)]


class _Diag(ctypes.Structure):
    _fields_ = [("have", _P), ("far_den", _P), ("far_abs", _P), ("den", _P)]


def load_library(path: str):
    """Load a compiled oracle (the default one, or a test's planted-mistake copy)."""
    lib = ctypes.CDLL(path)
    lib.oo_init.argtypes = [ctypes.POINTER(_Geom), _P, ctypes.c_int64, ctypes.POINTER(_State)]
    lib.oo_init.restype = None
    lib.oo_rows.argtypes = [ctypes.POINTER(_Geom), ctypes.POINTER(_State), _P, _P, _P, _P,
                            ctypes.c_int32, _P, ctypes.POINTER(_Diag), ctypes.c_int32]
    lib.oo_rows.restype = ctypes.c_int32
    lib.oo_back.argtypes = [ctypes.POINTER(_Geom), ctypes.POINTER(_State), ctypes.c_int32]
    lib.oo_back.restype = ctypes.c_int32
    lib.oo_rope.argtypes = [ctypes.c_int32, ctypes.c_int64, ctypes.c_float, _P, _P]
    lib.oo_rope.restype = None
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(build())
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


@dataclass
class Geom:
    """Layer shape. ``window`` is the ring stride (the widest group window)."""
    groups: int
    heads_per_group: int
    d: int
    dv: int
    sinks: int
    window: int
    landmarks: int
    scale: float | None = None
    rope_base: float = 1e6
    rect_far_mass: bool = False

    @property
    def nh(self) -> int:
        return self.groups * self.heads_per_group

    def scale_f32(self) -> float:
        s = self.scale if self.scale is not None else 1.0 / np.sqrt(self.d)
        return float(np.float32(s))

    def _c(self) -> _Geom:
        return _Geom(self.groups, self.heads_per_group, self.d, self.dv, self.sinks,
                     self.window, self.landmarks, int(bool(self.rect_far_mass)),
                     self.scale_f32(), float(np.float32(self.rope_base)))


def rope(x: np.ndarray, pos: int, base: float, lib=None) -> np.ndarray:
    """Rotate one head vector ``x`` (f32, length d) at position ``pos``."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape[0], dtype=np.float64)
    (lib or _load()).oo_rope(x.shape[0], int(pos), float(np.float32(base)), _ptr(x), _ptr(out))
    return out


class OracleLayer:
    """One sealed layer's state, held in double, advanced one row at a time."""

    def __init__(self, geom: Geom, sink_k, sink_v, k_tilde, q_tilde, mu,
                 group_windows=None, pos0: int = 0, lib=None):
        self._lib = lib or _load()
        g = geom
        self.geom = g
        G, hpg, nh, m = g.groups, g.heads_per_group, g.nh, g.landmarks
        f64 = lambda a, shape: np.ascontiguousarray(np.asarray(a, dtype=np.float32), dtype=np.float64).reshape(shape)
        self.meta = np.zeros((G, 4), dtype=np.int32)
        self.pos = np.zeros(1, dtype=np.int64)
        self.ring_k = np.zeros((G, g.window, g.d))
        self.ring_v = np.zeros((G, g.window, g.dv))
        self.sink_k = f64(sink_k, (G, g.sinks, g.d))
        self.sink_v = f64(sink_v, (G, g.sinks, g.dv))
        self.kt = f64(k_tilde, (G, m, g.d))
        self.qt = f64(q_tilde, (G, hpg, m, g.d))
        self.mu = f64(mu, (nh, m, m))
        self.M = np.zeros((nh, m))
        self.Z = np.zeros((nh, m))
        self.T = np.zeros((nh, m, g.dv))
        gw = None
        if group_windows is not None:
            gw = np.ascontiguousarray(group_windows, dtype=np.int32)
            assert gw.shape == (G,) and (gw <= g.window).all()
        self._g = g._c()
        self._st = _State(*[_ptr(a) for a in (self.meta, self.pos, self.ring_k, self.ring_v,
                                              self.sink_k, self.sink_v, self.kt, self.qt,
                                              self.mu, self.M, self.Z, self.T)])
        self._lib.oo_init(ctypes.byref(self._g), _ptr(gw), int(pos0), ctypes.byref(self._st))
        self.threads_used = 1

    def rows(self, q, k, v, gate=None, threads: int = 1, diag: bool = False):
        """Advance by ``rows`` rows; returns out [rows][nh][dv] (float64), and
        with ``diag`` also (have, far_den, far_abs, den) per (row, head)."""
        g = self.geom
        q = np.ascontiguousarray(q, dtype=np.float32)
        rows = q.shape[0]
        q = q.reshape(rows, g.nh, g.d)
        k = np.ascontiguousarray(k, dtype=np.float32).reshape(rows, g.groups, g.d)
        v = np.ascontiguousarray(v, dtype=np.float32).reshape(rows, g.groups, g.dv)
        if gate is not None:
            gate = np.ascontiguousarray(gate, dtype=np.float32).reshape(rows, g.nh, g.dv)
        out = np.empty((rows, g.nh, g.dv))
        dg = None
        dgp = None
        if diag:
            dg = (np.zeros((rows, g.nh), dtype=np.int8), np.zeros((rows, g.nh)), np.zeros((rows, g.nh)),
                  np.zeros((rows, g.nh)))
            dgp = ctypes.byref(_Diag(*[_ptr(a) for a in dg]))
        if rows > 0:
            self.threads_used = self._lib.oo_rows(ctypes.byref(self._g), ctypes.byref(self._st),
                                                _ptr(q), _ptr(k), _ptr(v), _ptr(gate), rows,
                                                _ptr(out), dgp, int(threads))
        return (out, dg) if diag else out

    def back(self, rows: int) -> bool:
        """Rewind ``rows`` ring pushes (meta and position only); False, with
        nothing changed, when a group cannot rewind that far."""
        return self._lib.oo_back(ctypes.byref(self._g), ctypes.byref(self._st), int(rows)) == 0

    def snapshot(self) -> dict:
        """The mutable state, copied: meta, pos, ring, far field."""
        return {"meta": self.meta.copy(), "pos": int(self.pos[0]), "ring_k": self.ring_k.copy(),
                "ring_v": self.ring_v.copy(), "M": self.M.copy(), "Z": self.Z.copy(),
                "T": self.T.copy()}
