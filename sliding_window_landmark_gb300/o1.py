"""Thin ctypes binding of the C ABI in include/o1.h (libo1.so).

Argument marshalling only: every function has the C name, passes pointers
and sizes through unchanged and returns the C status code (``check`` turns
a non-zero status into an exception). Device arguments are torch CUDA
tensors; their device, dtype, contiguity and size are checked here so that a
host pointer is never handed to a kernel. Every step of the computation runs
in the library's CUDA kernels; there is no other implementation to fall back
to, and importing this module fails if the library is not built.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

O1_OK = 0
O1_ERR_ARG = -1
O1_ERR_UNSUPPORTED = -2
O1_ERR_CUDA = -3
O1_ERR_STATE = -4


class O1Error(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        super().__init__(f"{what}: status {status} ({o1_status_string(status)})")
        self.status = status


class o1_geom(ctypes.Structure):
    _fields_ = [("groups", ctypes.c_int32), ("heads_per_group", ctypes.c_int32),
                ("d", ctypes.c_int32), ("dv", ctypes.c_int32), ("sinks", ctypes.c_int32),
                ("window", ctypes.c_int32), ("landmarks", ctypes.c_int32),
                ("rect_far_mass", ctypes.c_int32), ("scale", ctypes.c_float),
                ("rope_base", ctypes.c_float)]

    @property
    def nh(self) -> int:
        return self.groups * self.heads_per_group


class o1_state_host(ctypes.Structure):
    _fields_ = [("meta", ctypes.c_void_p), ("pos", ctypes.c_void_p), ("ring_k", ctypes.c_void_p),
                ("ring_v", ctypes.c_void_p), ("far_max", ctypes.c_void_p),
                ("far_mass", ctypes.c_void_p), ("far_val", ctypes.c_void_p)]


_VP = ctypes.c_void_p
_G = ctypes.POINTER(o1_geom)


def _load(path: str | None = None):
    path = path or _build.LIB
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -m sliding_window_landmark_gb300.build`")
    lib = ctypes.CDLL(path)
    lib.o1_state_bytes.argtypes = [_G]
    lib.o1_state_bytes.restype = ctypes.c_size_t
    lib.o1_scratch_bytes.argtypes = [_G, ctypes.c_int32]
    lib.o1_scratch_bytes.restype = ctypes.c_size_t
    lib.o1_state_init.argtypes = [_VP, _G, _VP, _VP, _VP, _VP, _VP, _VP, ctypes.c_int64, _VP]
    lib.o1_state_init.restype = ctypes.c_int
    lib.o1_chunk_attend.argtypes = [_VP, _G, _VP, ctypes.c_size_t, _VP, _VP, _VP, _VP, ctypes.c_int32, _VP, _VP]
    lib.o1_chunk_attend.restype = ctypes.c_int
    lib.o1_chunk_attend_timed.argtypes = [_VP, _G, _VP, ctypes.c_size_t, _VP, _VP, _VP, _VP, ctypes.c_int32,
                                          _VP, ctypes.POINTER(_VP), ctypes.c_int32, _VP]
    lib.o1_chunk_attend_timed.restype = ctypes.c_int
    lib.o1_chunk_attend_spec.argtypes = [_VP, _G, _VP, ctypes.c_size_t, _VP, _VP, _VP, _VP, ctypes.c_int32, _VP,
                                         _VP]
    lib.o1_chunk_attend_spec.restype = ctypes.c_int
    lib.o1_spec_commit.argtypes = [_VP, _G, _VP, ctypes.c_size_t, _VP, _VP, ctypes.c_int32, _VP]
    lib.o1_spec_commit.restype = ctypes.c_int
    lib.o1_window_attend.argtypes = [_VP, _G, _VP, ctypes.c_size_t, _VP, _VP, _VP, _VP, ctypes.c_int32, _VP, _VP]
    lib.o1_window_attend.restype = ctypes.c_int
    lib.o1_state_back.argtypes = [_VP, _G, ctypes.c_int32, _VP]
    lib.o1_state_back.restype = ctypes.c_int
    lib.o1_stage_name.argtypes = [ctypes.c_int32]
    lib.o1_stage_name.restype = ctypes.c_char_p
    lib.o1_token_attend.argtypes = [_VP, _G, _VP, ctypes.c_size_t, _VP, _VP, _VP, _VP, _VP, _VP]
    lib.o1_token_attend.restype = ctypes.c_int
    lib.o1_token_attend_noalloc.argtypes = [_VP, _G, _VP, _VP, _VP, _VP, _VP, _VP]
    lib.o1_token_attend_noalloc.restype = ctypes.c_int
    lib.o1_state_read.argtypes = [_VP, _G, ctypes.POINTER(o1_state_host), _VP]
    lib.o1_state_read.restype = ctypes.c_int
    lib.o1_state_write.argtypes = [_VP, _G, ctypes.POINTER(o1_state_host), _VP]
    lib.o1_state_write.restype = ctypes.c_int
    lib.o1_state_flags.argtypes = [_VP, _G, ctypes.POINTER(ctypes.c_uint32), ctypes.c_int32, _VP]
    lib.o1_state_flags.restype = ctypes.c_int
    lib.o1_status_string.argtypes = [ctypes.c_int]
    lib.o1_status_string.restype = ctypes.c_char_p
    lib.o1_set_wait_limit.argtypes = [ctypes.c_int64]
    lib.o1_set_wait_limit.restype = ctypes.c_int
    return lib


def _header_defines(names):
    """Integer #defines of include/o1.h (unsigned suffixes dropped), so that
    the binding's constants are the header's and cannot drift from them."""
    import re
    text = open(os.path.join(_build.INCLUDE, "o1.h")).read()
    out = {}
    for n in names:
        m = re.search(r"^#define\s+" + n + r"\s+(.+?)\s*(/\*.*)?$", text, re.M)
        if not m:
            raise RuntimeError(f"{n} is not defined in include/o1.h")
        expr = re.sub(r"(\d+)[uU]", r"\1", m.group(1))
        if not re.fullmatch(r"[\d\s()<>|+*x]+", expr):
            raise RuntimeError(f"{n}: unexpected definition {expr!r}")
        out[n] = int(eval(expr, {"__builtins__": {}}))
    return out


_DEF = _header_defines(["O1_NUM_STAGES", "O1_NOALLOC_SCRATCH_BYTES", "O1_FLAG_WAIT_EXPIRED",
                        "O1_FLAG_FP16_RANGE", "O1_FLAG_BACK_REFUSED"])


LIB = _load()
LIB_PATH = _build.LIB


def geom(groups: int, heads_per_group: int, d: int, dv: int, sinks: int, window: int, landmarks: int,
         scale: float | None = None, rope_base: float = 1e6, rect_far_mass: bool = False) -> o1_geom:
    """An o1_geom (scale defaults to 1/sqrt(d), rounded to f32)."""
    if scale is None:
        scale = 1.0 / d ** 0.5
    return o1_geom(groups, heads_per_group, d, dv, sinks, window, landmarks, int(bool(rect_far_mass)),
                   float(scale), float(rope_base))


def check(status: int, what: str = "o1") -> None:
    if status != O1_OK:
        raise O1Error(status, what)


def _dev(t, numel: int | None = None, name: str = "", dtype=torch.float32):
    """A device pointer from a CUDA tensor (None -> NULL)."""
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name}: expected a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: tensor must be contiguous")
    if numel is not None and t.numel() * t.element_size() < numel * (4 if dtype is not None else 1):
        raise ValueError(f"{name}: buffer too small ({t.numel()} elements, need {numel})")
    return _VP(t.data_ptr())


def _stream(stream):
    if stream is None:
        return _VP(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return _VP(stream.cuda_stream)
    return _VP(int(stream))


def o1_status_string(status: int) -> str:
    return LIB.o1_status_string(int(status)).decode()


def o1_state_bytes(g: o1_geom) -> int:
    return int(LIB.o1_state_bytes(ctypes.byref(g)))


def o1_scratch_bytes(g: o1_geom, max_rows: int) -> int:
    return int(LIB.o1_scratch_bytes(ctypes.byref(g), int(max_rows)))


def o1_state_init(state, g: o1_geom, group_windows, sink_k, sink_v, k_tilde, q_tilde, mu,
                  pos0: int = 0, stream=None) -> int:
    G, nh, m = g.groups, g.nh, g.landmarks
    gw = None
    if group_windows is not None:
        arr = (ctypes.c_int32 * G)(*[int(x) for x in group_windows])
        gw = ctypes.cast(arr, _VP)
    return LIB.o1_state_init(
        _dev(state, o1_state_bytes(g), "state", dtype=None), ctypes.byref(g), gw,
        _dev(sink_k, G * g.sinks * g.d, "sink_k"), _dev(sink_v, G * g.sinks * g.dv, "sink_v"),
        _dev(k_tilde, G * m * g.d, "k_tilde"), _dev(q_tilde, nh * m * g.d, "q_tilde"),
        _dev(mu, nh * m * m, "mu"), int(pos0), _stream(stream))


def o1_chunk_attend(state, g: o1_geom, scratch, q, k, v, gate, rows: int, out, stream=None) -> int:
    nh, G = g.nh, g.groups
    return LIB.o1_chunk_attend(
        _dev(state, None, "state", dtype=None), ctypes.byref(g), _dev(scratch, None, "scratch", dtype=None),
        scratch.numel() * scratch.element_size(),
        _dev(q, rows * nh * g.d, "q"), _dev(k, rows * G * g.d, "k"), _dev(v, rows * G * g.dv, "v"),
        _dev(gate, rows * nh * g.dv, "gate"), int(rows), _dev(out, rows * nh * g.dv, "out"), _stream(stream))


def o1_chunk_attend_spec(state, g: o1_geom, scratch, q, k, v, gate, rows: int, out, stream=None) -> int:
    """Attend ``rows`` draft rows without moving the state."""
    nh, G = g.nh, g.groups
    return LIB.o1_chunk_attend_spec(
        _dev(state, None, "state", dtype=None), ctypes.byref(g), _dev(scratch, None, "scratch", dtype=None),
        scratch.numel() * scratch.element_size(),
        _dev(q, rows * nh * g.d, "q"), _dev(k, rows * G * g.d, "k"), _dev(v, rows * G * g.dv, "v"),
        _dev(gate, rows * nh * g.dv, "gate"), int(rows), _dev(out, rows * nh * g.dv, "out"), _stream(stream))


def o1_spec_commit(state, g: o1_geom, scratch, k, v, rows: int, stream=None) -> int:
    """Move the state over the first ``rows`` accepted rows (their k and v)."""
    G = g.groups
    return LIB.o1_spec_commit(
        _dev(state, None, "state", dtype=None), ctypes.byref(g), _dev(scratch, None, "scratch", dtype=None),
        scratch.numel() * scratch.element_size(),
        _dev(k, rows * G * g.d, "k"), _dev(v, rows * G * g.dv, "v"), int(rows), _stream(stream))


def o1_window_attend(state, g: o1_geom, scratch, q, k, v, gate, rows: int, out, stream=None) -> int:
    """Exact sliding-window attention (sinks + window, no far field), attend only."""
    nh, G = g.nh, g.groups
    return LIB.o1_window_attend(
        _dev(state, None, "state", dtype=None), ctypes.byref(g), _dev(scratch, None, "scratch", dtype=None),
        scratch.numel() * scratch.element_size(),
        _dev(q, rows * nh * g.d, "q"), _dev(k, rows * G * g.d, "k"), _dev(v, rows * G * g.dv, "v"),
        _dev(gate, rows * nh * g.dv, "gate"), int(rows), _dev(out, rows * nh * g.dv, "out"), _stream(stream))


def o1_state_back(state, g: o1_geom, rows: int, stream=None) -> int:
    """Rewind the last ``rows`` ring pushes (meta and position)."""
    return LIB.o1_state_back(_dev(state, None, "state", dtype=None), ctypes.byref(g), int(rows), _stream(stream))


O1_NUM_STAGES = _DEF["O1_NUM_STAGES"]


def o1_stage_name(stage: int):
    n = LIB.o1_stage_name(int(stage))
    return None if n is None else n.decode()


def o1_chunk_attend_timed(state, g: o1_geom, scratch, q, k, v, gate, rows: int, out, events, stream=None) -> int:
    """``events``: 2 * O1_NUM_STAGES torch.cuda.Event(enable_timing=True),
    each already recorded once (so that its CUDA handle exists); stage i's
    time is events[2i].elapsed_time(events[2i + 1])."""
    nh, G = g.nh, g.groups
    arr = (_VP * len(events))(*[_VP(int(e.cuda_event)) for e in events])
    return LIB.o1_chunk_attend_timed(
        _dev(state, None, "state", dtype=None), ctypes.byref(g), _dev(scratch, None, "scratch", dtype=None),
        scratch.numel() * scratch.element_size(),
        _dev(q, rows * nh * g.d, "q"), _dev(k, rows * G * g.d, "k"), _dev(v, rows * G * g.dv, "v"),
        _dev(gate, rows * nh * g.dv, "gate"), int(rows), _dev(out, rows * nh * g.dv, "out"), arr, len(events),
        _stream(stream))


def o1_token_attend(state, g: o1_geom, scratch, q, k, v, gate, out, stream=None) -> int:
    nh, G = g.nh, g.groups
    return LIB.o1_token_attend(
        _dev(state, None, "state", dtype=None), ctypes.byref(g), _dev(scratch, None, "scratch", dtype=None),
        scratch.numel() * scratch.element_size(),
        _dev(q, nh * g.d, "q"), _dev(k, G * g.d, "k"), _dev(v, G * g.dv, "v"),
        _dev(gate, nh * g.dv, "gate"), _dev(out, nh * g.dv, "out"), _stream(stream))


O1_NOALLOC_SCRATCH_BYTES = _DEF["O1_NOALLOC_SCRATCH_BYTES"]


def o1_token_attend_noalloc(state, g: o1_geom, q, k, v, gate, out, stream=None) -> int:
    """o1_token_attend without a scratch argument: the library's own static
    device scratch is used (see include/o1.h)."""
    nh, G = g.nh, g.groups
    return LIB.o1_token_attend_noalloc(
        _dev(state, None, "state", dtype=None), ctypes.byref(g),
        _dev(q, nh * g.d, "q"), _dev(k, G * g.d, "k"), _dev(v, G * g.dv, "v"),
        _dev(gate, nh * g.dv, "gate"), _dev(out, nh * g.dv, "out"), _stream(stream))


def _host_view(g: o1_geom, arrays: dict):
    """An o1_state_host over numpy arrays (missing keys -> NULL)."""
    import numpy as np
    want = {"meta": (np.uint32, g.groups * 4), "pos": (np.int64, 1),
            "ring_k": (np.float32, g.groups * g.window * g.d), "ring_v": (np.float32, g.groups * g.window * g.dv),
            "far_max": (np.float32, g.nh * g.landmarks), "far_mass": (np.float32, g.nh * g.landmarks),
            "far_val": (np.float32, g.nh * g.landmarks * g.dv)}
    ptrs = {}
    for key, (dt, n) in want.items():
        a = arrays.get(key)
        if a is None:
            ptrs[key] = None
            continue
        if a.dtype != dt or not a.flags["C_CONTIGUOUS"] or a.size < n:
            raise ValueError(f"{key}: need a C-contiguous {dt.__name__} array of {n} elements")
        ptrs[key] = a.ctypes.data_as(_VP)
    return o1_state_host(**ptrs)


def o1_state_read(state, g: o1_geom, dst: dict, stream=None) -> int:
    """Fills the numpy arrays in ``dst`` (keys of o1_state_host)."""
    hv = _host_view(g, dst)
    return LIB.o1_state_read(_dev(state, o1_state_bytes(g), "state", dtype=None), ctypes.byref(g),
                             ctypes.byref(hv), _stream(stream))


def o1_state_write(state, g: o1_geom, src: dict, stream=None) -> int:
    hv = _host_view(g, src)
    return LIB.o1_state_write(_dev(state, o1_state_bytes(g), "state", dtype=None), ctypes.byref(g),
                              ctypes.byref(hv), _stream(stream))


O1_FLAG_WAIT_EXPIRED = _DEF["O1_FLAG_WAIT_EXPIRED"]
O1_FLAG_FP16_RANGE = _DEF["O1_FLAG_FP16_RANGE"]
O1_FLAG_BACK_REFUSED = _DEF["O1_FLAG_BACK_REFUSED"]


def o1_set_wait_limit(cycles: int) -> int:
    """Limit of the kernels' first waits for later calls (cycles < 1: the default)."""
    return LIB.o1_set_wait_limit(int(cycles))


def o1_state_flags(state, g: o1_geom, clear: bool = False, stream=None) -> int:
    """The state's sticky flags (O1_FLAG_*); raises O1Error on a bad status."""
    f = ctypes.c_uint32(0)
    check(LIB.o1_state_flags(_dev(state, o1_state_bytes(g), "state", dtype=None), ctypes.byref(g),
                             ctypes.byref(f), int(bool(clear)), _stream(stream)), "flags")
    return int(f.value)


def empty_state_arrays(g: o1_geom) -> dict:
    """Host arrays for every part o1_state_read can fill."""
    import numpy as np
    return {"meta": np.zeros((g.groups, 4), np.uint32), "pos": np.zeros(1, np.int64),
            "ring_k": np.zeros((g.groups, g.window, g.d), np.float32),
            "ring_v": np.zeros((g.groups, g.window, g.dv), np.float32),
            "far_max": np.zeros((g.nh, g.landmarks), np.float32),
            "far_mass": np.zeros((g.nh, g.landmarks), np.float32),
            "far_val": np.zeros((g.nh, g.landmarks, g.dv), np.float32)}
