"""The C-ABI library without a GPU: it loads, exports every entry point that
include/o1.h declares, sizes buffers on the host, and rejects bad arguments
before any CUDA call (so nothing here touches a device)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def o1():
    from sliding_window_landmark_gb300 import build
    build.build()
    from sliding_window_landmark_gb300 import o1 as mod
    return mod


def declared_entry_points():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"O1_API\s+[\w\s\*]*?\b(o1_\w+)\s*\(", text)
    return names


def test_every_declared_symbol_is_exported(o1):
    names = declared_entry_points()
    assert {"o1_state_init", "o1_chunk_attend", "o1_token_attend", "o1_state_read"} <= set(names)
    lib = ctypes.CDLL(o1.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n


def test_sizes(o1):
    g = o1.geom(2, 4, 256, 256, 4, 2048, 32)
    sb = o1.o1_state_bytes(g)
    # ring K+V dominates: 2 groups x 2048 x 512 floats
    assert 2 * 2048 * 512 * 4 < sb < 2 * 2048 * 512 * 4 + 2_000_000
    s1, s64, s4096 = (o1.o1_scratch_bytes(g, n) for n in (1, 64, 4096))
    assert 0 < s1 <= s64 < s4096
    assert o1.o1_scratch_bytes(g, 0) == 0
    for bad in (o1.geom(0, 4, 256, 256, 4, 2048, 32), o1.geom(2, 4, 260, 256, 4, 2048, 32),
                o1.geom(2, 4, 256, 256, 4, 2048, 65), o1.geom(2, 17, 256, 256, 4, 2048, 32),
                o1.geom(2, 4, 12, 12, 4, 2048, 32), o1.geom(2, 4, 256, 256, 65, 2048, 32)):
        assert o1.o1_state_bytes(bad) == 0


def test_scratch_grows_with_rows(o1):
    """The library finds a scratch's row capacity by bisection, so the bytes
    it needs must not shrink as rows grow."""
    for g in (o1.geom(2, 4, 256, 256, 4, 2048, 32), o1.geom(4, 4, 128, 128, 4, 1024, 64),
              o1.geom(1, 2, 64, 64, 4, 16, 4), o1.geom(3, 16, 72, 20, 0, 40, 1)):
        sizes = [o1.o1_scratch_bytes(g, r) for r in list(range(1, 300)) + [1000, 4096, 4097]]
        assert all(b >= a for a, b in zip(sizes, sizes[1:]))


def test_validation_before_any_launch(o1):
    L = o1.LIB
    g = o1.geom(1, 2, 64, 64, 4, 16, 4)
    gp = ctypes.byref(g)
    V = ctypes.c_void_p
    aligned = V(1 << 20)
    # unsupported geometry
    bad = o1.geom(1, 2, 63, 64, 4, 16, 4)
    assert L.o1_chunk_attend(aligned, ctypes.byref(bad), aligned, 1 << 20, aligned, aligned, aligned, None, 4,
                             aligned, None) == o1.O1_ERR_UNSUPPORTED
    # null buffers
    assert L.o1_chunk_attend(None, gp, aligned, 1 << 20, aligned, aligned, aligned, None, 4, aligned,
                             None) == o1.O1_ERR_ARG
    assert L.o1_chunk_attend(aligned, gp, aligned, 1 << 20, None, aligned, aligned, None, 4, aligned,
                             None) == o1.O1_ERR_ARG
    # negative rows; zero rows is a no-op
    assert L.o1_chunk_attend(aligned, gp, aligned, 1 << 20, aligned, aligned, aligned, None, -1, aligned,
                             None) == o1.O1_ERR_ARG
    assert L.o1_chunk_attend(aligned, gp, aligned, 1 << 20, aligned, aligned, aligned, None, 0, aligned,
                             None) == o1.O1_OK
    # misaligned state / inputs
    assert L.o1_chunk_attend(V((1 << 20) + 16), gp, aligned, 1 << 20, aligned, aligned, aligned, None, 4,
                             V(1 << 22), None) == o1.O1_ERR_ARG
    assert L.o1_chunk_attend(aligned, gp, aligned, 1 << 20, V((1 << 21) + 4), aligned, aligned, None, 4,
                             V(1 << 22), None) == o1.O1_ERR_ARG
    # scratch too small for even one row
    assert L.o1_chunk_attend(aligned, gp, aligned, 16, V(1 << 21), V(1 << 21), V(1 << 21), None, 4,
                             V(1 << 23), None) == o1.O1_ERR_ARG
    # out overlapping an input
    assert L.o1_chunk_attend(aligned, gp, aligned, 1 << 20, V(1 << 21), V(1 << 22), V(1 << 23), None, 4,
                             V(1 << 21), None) == o1.O1_ERR_ARG
    # token path: same checks
    assert L.o1_token_attend(None, gp, aligned, 1 << 20, aligned, aligned, aligned, None, aligned,
                             None) == o1.O1_ERR_ARG
    # speculative pair: attend-only drafts must fit one pass; commit checks its own buffers
    assert L.o1_chunk_attend_spec(None, gp, aligned, 1 << 20, aligned, aligned, aligned, None, 4, aligned,
                                  None) == o1.O1_ERR_ARG
    assert L.o1_chunk_attend_spec(aligned, gp, aligned, 1 << 20, V(1 << 24), V(1 << 26), V(1 << 28), None,
                                  1 << 16, V(1 << 30), None) == o1.O1_ERR_ARG
    assert L.o1_spec_commit(aligned, gp, aligned, 1 << 20, aligned, aligned, 0, None) == o1.O1_OK
    assert L.o1_spec_commit(aligned, gp, aligned, 1 << 20, aligned, aligned, -1, None) == o1.O1_ERR_ARG
    assert L.o1_spec_commit(aligned, gp, aligned, 1 << 20, None, aligned, 4, None) == o1.O1_ERR_ARG
    assert L.o1_spec_commit(aligned, gp, aligned, 1 << 20, aligned, V((1 << 21) + 8), 4, None) == o1.O1_ERR_ARG
    assert L.o1_spec_commit(aligned, gp, aligned, 16, aligned, aligned, 4, None) == o1.O1_ERR_ARG
    assert L.o1_spec_commit(aligned, ctypes.byref(bad), aligned, 1 << 20, aligned, aligned, 4,
                            None) == o1.O1_ERR_UNSUPPORTED
    # comparator: same checks; attend-only, so one pass
    assert L.o1_window_attend(None, gp, aligned, 1 << 20, aligned, aligned, aligned, None, 4, aligned,
                              None) == o1.O1_ERR_ARG
    assert L.o1_window_attend(aligned, gp, aligned, 1 << 20, V(1 << 24), V(1 << 26), V(1 << 28), None,
                              1 << 16, V(1 << 30), None) == o1.O1_ERR_ARG
    # rewind: checks before any launch; zero rows is a no-op
    assert L.o1_state_back(None, gp, 1, None) == o1.O1_ERR_ARG
    assert L.o1_state_back(V((1 << 20) + 16), gp, 1, None) == o1.O1_ERR_ARG
    assert L.o1_state_back(aligned, gp, -1, None) == o1.O1_ERR_ARG
    assert L.o1_state_back(aligned, gp, 0, None) == o1.O1_OK
    assert L.o1_state_back(aligned, ctypes.byref(bad), 1, None) == o1.O1_ERR_UNSUPPORTED
    # init: bad group window, missing landmarks
    gw = (ctypes.c_int32 * 1)(17)
    assert L.o1_state_init(aligned, gp, ctypes.cast(gw, V), aligned, aligned, aligned, aligned, aligned, 0,
                           None) == o1.O1_ERR_ARG
    assert L.o1_state_init(aligned, gp, None, aligned, aligned, None, aligned, aligned, 0, None) == o1.O1_ERR_ARG
    assert L.o1_state_init(aligned, gp, None, aligned, aligned, aligned, aligned, aligned, -5, None) == o1.O1_ERR_ARG
    assert o1.o1_status_string(o1.O1_ERR_STATE).startswith("state header")
