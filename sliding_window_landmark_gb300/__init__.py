"""Sealed O(1) layer attention (sinks + ring-buffer window + landmark far
field) for GB300, as hand-written sm_103a CUDA behind a C ABI.

``sliding_window_landmark_gb300.o1`` is the thin ctypes binding of the C ABI
declared in ``include/o1.h``; ``synth`` makes seeded synthetic inputs.
"""
from . import synth  # noqa: F401

__all__ = ["synth", "o1"]


def __getattr__(name):
    if name == "o1":
        import importlib
        return importlib.import_module(".o1", __name__)
    raise AttributeError(name)
