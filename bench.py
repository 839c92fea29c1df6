#!/usr/bin/env python
"""Benchmark of the sealed O(1) layer hot path on one GB300 (per rank).

Workload: one Qwen3.5-0.8B-shaped sealed layer (2 KV groups x 4 query heads,
d = dv = 256, 4 sinks, window 2048, 32 landmarks per head, rotary base 1e6,
sigmoid output gate), a 4096-row prompt from a fresh state, processed by one
o1_chunk_attend call. One step = restore the fresh state (device copy) + the
call. Inputs are seeded N(0,1) (synthetic). Three rotating input sets keep
each step's inputs out of L2 (their total is well above the 129 MB L2).

Prints one JSON line: prefill rows/s (whole job over all ranks), the dominant
kernel against its roofline, the oracle on the host cores, the end-to-end
rate with host buffers, clocks, and beside them: decode us/token after an
8192-row prompt (`decode`) and across a 24-layer stack whose states exceed
L2 (`decode_stack`), both against HBM; exact causal attention over the same
prompt (`comparator`); speculative verify + commit cycles (`speculative`);
ring rewinds (`rewind`).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from sliding_window_landmark_gb300 import synth  # noqa: E402

SHAPE = synth.QWEN_LAYER
SEED = 1
ROWS = 4096
DECODE_PREFILL = 8192
DECODE_STEPS = 256
SPEC_DRAFT, SPEC_ACC, SPEC_CYCLES = 8, 5, 64
STACK_LAYERS, STACK_PREFILL, STACK_STEPS = 24, 1100, 32
N_SETS = 3
WORKLOAD = ("Qwen3.5-0.8B-shaped sealed layer: G=2 KV groups x 4 query heads, d=dv=256, 4 sinks, "
            "window 2048, 32 landmarks/head, rope base 1e6, sigmoid gate; 4096-row prompt from a fresh "
            "state in one o1_chunk_attend call (64-row far-field blocks)")
METRIC = "sealed-layer prefill rows/s"
FP32_PEAK_TFLOPS = 152 * 128 * 2 * 2.070e9 / 1e12   # SMs x FP32 lanes x 2 flop x max SM clock


# ------------------------------------------------------------------ helpers

def window_flops(shape: synth.Shape, rows: int, len0: int = 0) -> float:
    """Algorithmic flops of the window attention: 2 window_r (d + dv) per
    row-head (q.k and p.v over the row's window keys),
    window_r = min(wg, len0 + r + 1)."""
    wins = shape.group_windows or (shape.window,) * shape.groups
    r = np.arange(rows)
    tot = 0.0
    for wg in wins:
        tot += shape.heads_per_group * float(np.sum(2.0 * np.minimum(wg, len0 + r + 1) * (shape.d + shape.dv)))
    return tot


def tensor_core_window(shape: synth.Shape) -> bool:
    return shape.d % 64 == 0 and shape.d <= 256 and shape.dv % 32 == 0 and shape.dv <= 256 and shape.window >= 512


def decode_bytes(shape: synth.Shape) -> float:
    """Bytes one decode step must move: the whole state once (ring K and V,
    landmark queries/keys, mu, sinks, far max/mass), the far value sum read
    and written, and the row's inputs and output."""
    G, nh, d, dv, w, m, ns = shape.groups, shape.nh, shape.d, shape.dv, shape.window, shape.landmarks, shape.sinks
    state = G * w * (d + dv) + nh * m * d + G * m * d + nh * m * m + G * ns * (d + dv) + 2 * nh * m
    far_val = 2 * nh * m * dv
    io = nh * d + G * (d + dv) + 2 * nh * dv
    return 4.0 * (state + far_val + io)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return j, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class Clocks:
    """Samples SM clock and clock-event reasons through NVML (read only)."""
    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap", 0x8: "hw_slowdown",
               0x10: "sync_boost", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting"}

    def __init__(self, torch_dev: int):
        self.ok = False
        self.samples, self.reasons = [], 0
        try:
            import torch
            self.nv = ctypes.CDLL("libnvidia-ml.so.1")
            assert self.nv.nvmlInit_v2() == 0
            self.h = ctypes.c_void_p()
            props = torch.cuda.get_device_properties(torch_dev)
            got = False
            bus = getattr(props, "pci_bus_id", None)
            if bus is not None:
                for s in (f"{getattr(props, 'pci_domain_id', 0):08X}:{bus:02X}:{getattr(props, 'pci_device_id', 0):02X}.0",
                          f"{getattr(props, 'pci_domain_id', 0):04X}:{bus:02X}:{getattr(props, 'pci_device_id', 0):02X}.0"):
                    if self.nv.nvmlDeviceGetHandleByPciBusId_v2(s.encode(), ctypes.byref(self.h)) == 0:
                        got = True
                        break
            if not got:
                assert self.nv.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(self.h)) == 0
            mx = ctypes.c_uint()
            self.nv.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx))
            self.max_mhz = int(mx.value)
            self.ok = True
        except Exception:
            self.ok = False

    def _sample(self):
        c, r = ctypes.c_uint(), ctypes.c_ulonglong()
        self.nv.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(c))
        fn = getattr(self.nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.nv.nvmlDeviceGetCurrentClocksThrottleReasons
        fn(self.h, ctypes.byref(r))
        self.samples.append(int(c.value))
        self.reasons |= int(r.value)

    def __enter__(self):
        self._stop = threading.Event()

        def run():
            while not self._stop.is_set():
                self._sample()
                time.sleep(0.002)
        if self.ok:
            self._sample()
            self._t = threading.Thread(target=run, daemon=True)
            self._t.start()
        return self

    def __exit__(self, *a):
        if self.ok:
            self._stop.set()
            self._t.join()
            self._sample()

    def summary(self):
        if not self.ok or not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvml unavailable"]}
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": [n for b, n in self.REASONS.items() if self.reasons & b], "samples": len(self.samples)}


def traffic_record(kernel: str):
    """ncu DRAM bytes of `kernel` per launch on this workload, if the committed
    record was taken from the current kernel source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f).get(kernel)
    if not rec:
        return None
    src = os.path.join(ROOT, rec["source"])
    if not os.path.exists(src) or hashlib.sha256(open(src, "rb").read()).hexdigest() != rec["sha256"]:
        return None
    return rec["dram_bytes_per_launch"]


# ------------------------------------------------------------ oracle timing

def oracle_prompt_rate(rows: int, threads: int):
    """The oracle, as it stands, over the first `rows` rows of the prompt."""
    import oracle
    c = synth.layer_constants(SHAPE, SEED)
    g = oracle.Geom(SHAPE.groups, SHAPE.heads_per_group, SHAPE.d, SHAPE.dv, SHAPE.sinks, SHAPE.window,
                    SHAPE.landmarks, rope_base=SHAPE.rope_base)
    lay = oracle.OracleLayer(g, c.sink_k, c.sink_v, c.k_tilde, c.q_tilde, c.mu)
    q, k, v, gt = synth.layer_rows(SHAPE, SEED, 0, rows)
    t0 = time.perf_counter()
    lay.rows(q, k, v, gt, threads=threads)
    dt = time.perf_counter() - t0
    return rows / dt, dt, lay.threads_used


def reference_arm(args, rank):
    """The oracle as the reference implementation, on the host cores: each
    step processes one 512-row slice of the same 4096-row prompt, restored
    from a snapshot taken at the slice's start during one untimed pass, so
    that 8 consecutive steps cover the whole prompt."""
    if rank != 0:
        return
    import oracle
    c = synth.layer_constants(SHAPE, SEED)
    g = oracle.Geom(SHAPE.groups, SHAPE.heads_per_group, SHAPE.d, SHAPE.dv, SHAPE.sinks, SHAPE.window,
                    SHAPE.landmarks, rope_base=SHAPE.rope_base)
    lay = oracle.OracleLayer(g, c.sink_k, c.sink_v, c.k_tilde, c.q_tilde, c.mu)
    q, k, v, gt = synth.layer_rows(SHAPE, SEED, 0, ROWS)
    slice_rows = 512
    snaps = []
    for s0 in range(0, ROWS, slice_rows):
        snaps.append({key: (val.copy() if isinstance(val, np.ndarray) else val)
                      for key, val in lay.snapshot().items()})
        lay.rows(q[s0:s0 + slice_rows], k[s0:s0 + slice_rows], v[s0:s0 + slice_rows], gt[s0:s0 + slice_rows],
                 threads=SHAPE.groups)

    def restore(i):
        s = snaps[i]
        lay.meta[...] = s["meta"]
        lay.pos[0] = s["pos"]
        lay.ring_k[...] = s["ring_k"]
        lay.ring_v[...] = s["ring_v"]
        lay.M[...] = s["M"]
        lay.Z[...] = s["Z"]
        lay.T[...] = s["T"]

    def step(i):
        j = i % len(snaps)
        restore(j)
        s0 = j * slice_rows
        lay.rows(q[s0:s0 + slice_rows], k[s0:s0 + slice_rows], v[s0:s0 + slice_rows], gt[s0:s0 + slice_rows],
                 threads=SHAPE.groups)
    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i)
    dt = time.perf_counter() - t0
    rate = slice_rows * args.steps / dt
    line = {"impl": "reference", "metric": METRIC, "value": rate, "unit": "rows/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "reference": "serial CPU oracle (plain C, double), rows serial, "
                       "KV groups on threads"},
            "cpu_baseline": {"value": rate, "unit": "rows/s", "cores": lay.threads_used, "kind": "oracle",
                             "sample": f"{slice_rows}-row slices of the 4096-row prompt, restored from "
                                       f"snapshots; {args.steps} slices timed"},
            "e2e": {"value": rate, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ our arm

def max_over_ranks(ms: float, world: int) -> float:
    """The slowest rank's time: every rank runs the same replica workload,
    so the job ends when the last one does (gloo all-reduce on the host)."""
    if world <= 1:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(rows_per_step: int, steps: int, world: int, ms_max: float) -> float:
    """Rows/s over all ranks: each rank processes its own rows (weak scaling)."""
    return rows_per_step * steps * world / (ms_max * 1e-3)


def our_arm(args, rank, world, local_rank):
    import torch
    from sliding_window_landmark_gb300 import build
    build.build()
    from sliding_window_landmark_gb300 import o1

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    sh = SHAPE
    g = o1.geom(sh.groups, sh.heads_per_group, sh.d, sh.dv, sh.sinks, sh.window, sh.landmarks,
                rope_base=sh.rope_base)
    c = synth.layer_constants(sh, SEED)
    up = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev)
    consts = [up(c.sink_k), up(c.sink_v), up(c.k_tilde), up(c.q_tilde), up(c.mu)]
    sbytes = o1.o1_state_bytes(g)
    pristine = torch.empty(sbytes, dtype=torch.uint8, device=dev)
    o1.check(o1.o1_state_init(pristine, g, None, *consts, 0), "init")
    scratch = torch.empty(o1.o1_scratch_bytes(g, ROWS), dtype=torch.uint8, device=dev)
    q, k, v, gt = synth.layer_rows(sh, SEED, 0, ROWS)
    hq, hk, hv, hg = (torch.from_numpy(x).pin_memory() for x in (q, k, v, gt))
    sets = []
    for i in range(N_SETS):
        sets.append({"q": hq.to(dev), "k": hk.to(dev), "v": hv.to(dev), "g": hg.to(dev),
                     "out": torch.empty((ROWS, sh.nh, sh.dv), dtype=torch.float32, device=dev),
                     "state": torch.empty(sbytes, dtype=torch.uint8, device=dev)})
    set_bytes = sum(t.numel() * t.element_size() for s in sets[:1] for t in s.values())

    nst = o1.O1_NUM_STAGES
    total_steps = args.warmup + args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * nst)] for _ in range(total_steps)]
    for row in evs:
        for e in row:
            e.record(stream)   # create the CUDA events before they are handed to the library
    torch.cuda.synchronize()

    def step(i):
        s = sets[i % N_SETS]
        s["state"].copy_(pristine, non_blocking=True)
        o1.check(o1.o1_chunk_attend_timed(s["state"], g, scratch, s["q"], s["k"], s["v"], s["g"], ROWS,
                                          s["out"], evs[i]), "chunk")

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    barrier()
    clk = Clocks(local_rank)
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with clk:
        torch.cuda.synchronize()
        t_start.record(stream)
        for i in range(args.steps):
            step(args.warmup + i)
        t_end.record(stream)
        torch.cuda.synchronize()
    barrier()
    ms = t_start.elapsed_time(t_end)
    stage_ms = [[evs[args.warmup + i][2 * j].elapsed_time(evs[args.warmup + i][2 * j + 1]) for j in range(nst)]
                for i in range(args.steps)]
    stage_avg = np.mean(np.array(stage_ms), axis=0)
    ms_max = max_over_ranks(ms, world)

    # parity spot check of the timed output against a fresh run (same inputs)
    out0 = sets[(args.warmup + args.steps - 1) % N_SETS]["out"]
    assert torch.isfinite(out0).all().item(), "non-finite output"

    # ---- end to end: host buffers in, host output back, through the C ABI
    host_out = torch.empty((ROWS, sh.nh, sh.dv), dtype=torch.float32).pin_memory()
    s = sets[0]

    def e2e_step():
        for name, h in (("q", hq), ("k", hk), ("v", hv), ("g", hg)):
            s[name].copy_(h, non_blocking=True)
        s["state"].copy_(pristine, non_blocking=True)
        o1.check(o1.o1_chunk_attend(s["state"], g, scratch, s["q"], s["k"], s["v"], s["g"], ROWS, s["out"]),
                 "chunk")
        host_out.copy_(s["out"], non_blocking=True)
    for _ in range(max(1, args.warmup)):
        e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hg))
    d2h = host_out.numel() * 4

    # ---- comparator: exact causal attention over the same 4096-row prompt
    # (window = the prompt, no sinks, no far field) through o1_window_attend,
    # the same window kernels, on the same rotating input sets
    gx = o1.geom(sh.groups, sh.heads_per_group, sh.d, sh.dv, 0, ROWS, sh.landmarks, rope_base=sh.rope_base)
    xstate = torch.empty(o1.o1_state_bytes(gx), dtype=torch.uint8, device=dev)
    o1.check(o1.o1_state_init(xstate, gx, None, None, None, consts[2], consts[3], consts[4], 0), "init")
    xscratch = torch.empty(o1.o1_scratch_bytes(gx, ROWS), dtype=torch.uint8, device=dev)

    def x_step(i):
        s = sets[i % N_SETS]
        o1.check(o1.o1_window_attend(xstate, gx, xscratch, s["q"], s["k"], s["v"], s["g"], ROWS, s["out"]), "exact")

    for i in range(args.warmup):
        x_step(i)
    torch.cuda.synchronize()
    x0, x1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    x0.record(stream)
    for i in range(args.steps):
        x_step(args.warmup + i)
    x1.record(stream)
    torch.cuda.synchronize()
    x_ms = x0.elapsed_time(x1) / args.steps
    x_flops = window_flops(synth.Shape(sh.groups, sh.heads_per_group, sh.d, sh.dv, 0, ROWS, sh.landmarks), ROWS)
    del xstate, xscratch

    # ---- decode: 8192-row prompt (untimed), then one-row steps
    dstate = torch.empty(sbytes, dtype=torch.uint8, device=dev)
    o1.check(o1.o1_state_init(dstate, g, None, *consts, 0), "init")
    dscratch = torch.empty(o1.o1_scratch_bytes(g, DECODE_PREFILL), dtype=torch.uint8, device=dev)
    pq, pk, pv, pg = (up(x) for x in synth.layer_rows(sh, 2, 0, DECODE_PREFILL))
    pout = torch.empty((DECODE_PREFILL, sh.nh, sh.dv), dtype=torch.float32, device=dev)
    o1.check(o1.o1_chunk_attend(dstate, g, dscratch, pq, pk, pv, pg, DECODE_PREFILL, pout), "prefill")
    del pq, pk, pv, pg, pout
    nd = args.warmup + DECODE_STEPS
    tq, tk, tv, tg = (up(x) for x in synth.layer_rows(sh, 2, DECODE_PREFILL, nd))
    tout = torch.empty((nd, sh.nh, sh.dv), dtype=torch.float32, device=dev)
    for i in range(args.warmup):
        o1.check(o1.o1_token_attend(dstate, g, dscratch, tq[i], tk[i], tv[i], tg[i], tout[i]), "token")
    torch.cuda.synchronize()
    # the 256 steps captured once as a CUDA graph (host launch cost out of the loop), then replayed
    graph = torch.cuda.CUDAGraph()
    cap_stream = torch.cuda.Stream()
    with torch.cuda.stream(cap_stream):
        with torch.cuda.graph(graph, stream=cap_stream):
            for i in range(args.warmup, nd):
                o1.check(o1.o1_token_attend(dstate, g, dscratch, tq[i], tk[i], tv[i], tg[i], tout[i]), "token")
    torch.cuda.synchronize()
    d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    d0.record(stream)
    graph.replay()
    d1.record(stream)
    torch.cuda.synchronize()
    dec_us = 1e3 * d0.elapsed_time(d1) / DECODE_STEPS
    dec_launches = 2

    # ---- speculative verify + commit on the same state: SPEC_DRAFT-row
    # drafts attended without moving the state, SPEC_ACC rows of each
    # committed; the cycles captured once as a CUDA graph and replayed
    sq, sk, sv, sg = (up(x) for x in synth.layer_rows(sh, 3, DECODE_PREFILL + nd, SPEC_DRAFT * (SPEC_CYCLES + 3)))
    sout = torch.empty((SPEC_DRAFT, sh.nh, sh.dv), dtype=torch.float32, device=dev)

    def spec_cycle(i):
        a, b = i * SPEC_DRAFT, (i + 1) * SPEC_DRAFT
        o1.check(o1.o1_chunk_attend_spec(dstate, g, dscratch, sq[a:b], sk[a:b], sv[a:b], sg[a:b], SPEC_DRAFT, sout),
                 "spec")
        o1.check(o1.o1_spec_commit(dstate, g, dscratch, sk[a:a + SPEC_ACC], sv[a:a + SPEC_ACC], SPEC_ACC), "commit")

    for i in range(3):
        spec_cycle(SPEC_CYCLES + i)
    torch.cuda.synchronize()
    sgraph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(cap_stream):
        with torch.cuda.graph(sgraph, stream=cap_stream):
            for i in range(SPEC_CYCLES):
                spec_cycle(i)
    torch.cuda.synchronize()
    d0.record(stream)
    sgraph.replay()
    d1.record(stream)
    torch.cuda.synchronize()
    spec_us = 1e3 * d0.elapsed_time(d1) / SPEC_CYCLES

    # ---- meta rewind: one-row rewinds then the same row pushed again by
    # o1_spec_commit, as a looped layer would, in one graph
    rk, rv = sk[:1], sv[:1]
    rgraph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(cap_stream):
        with torch.cuda.graph(rgraph, stream=cap_stream):
            for i in range(SPEC_CYCLES):
                o1.check(o1.o1_state_back(dstate, g, 1), "back")
                o1.check(o1.o1_spec_commit(dstate, g, dscratch, rk, rv, 1), "commit")
    torch.cuda.synchronize()
    d0.record(stream)
    rgraph.replay()
    d1.record(stream)
    torch.cuda.synchronize()
    back_us = 1e3 * d0.elapsed_time(d1) / SPEC_CYCLES
    assert o1.o1_state_flags(dstate, g) == 0, "state flags raised"
    dec_bytes = decode_bytes(sh)

    # ---- decode across a stack of STACK_LAYERS independent layers of the
    # stack shape, whose states together exceed L2: each layer prefilled past
    # its window (shared prompt rows, per-layer constants), then one-row steps
    # through every layer in turn, captured once in a CUDA graph
    ss = synth.STACK_LAYER
    gs = o1.geom(ss.groups, ss.heads_per_group, ss.d, ss.dv, ss.sinks, ss.window, ss.landmarks,
                 rope_base=ss.rope_base)
    sscr = torch.empty(o1.o1_scratch_bytes(gs, STACK_PREFILL), dtype=torch.uint8, device=dev)
    sp = [up(x) for x in synth.layer_rows(ss, 1000, 0, STACK_PREFILL)]
    st_rows = [up(x) for x in synth.layer_rows(ss, 1000, STACK_PREFILL, STACK_STEPS + 2)]
    pout = torch.empty((STACK_PREFILL, ss.nh, ss.dv), dtype=torch.float32, device=dev)
    sstates = []
    for layer in range(STACK_LAYERS):
        cl = synth.layer_constants(ss, 1000 + layer)
        cst = [up(cl.sink_k), up(cl.sink_v), up(cl.k_tilde), up(cl.q_tilde), up(cl.mu)]
        st_ = torch.empty(o1.o1_state_bytes(gs), dtype=torch.uint8, device=dev)
        o1.check(o1.o1_state_init(st_, gs, None, *cst, 0), "init")
        o1.check(o1.o1_chunk_attend(st_, gs, sscr, *sp, STACK_PREFILL, pout), "prefill")
        sstates.append(st_)
    del sp, pout
    sq_, sk_, sv_, sg_ = st_rows
    sout = torch.empty((ss.nh, ss.dv), dtype=torch.float32, device=dev)

    def stack_step(i):
        for st_ in sstates:
            o1.check(o1.o1_token_attend(st_, gs, sscr, sq_[i], sk_[i], sv_[i], sg_[i], sout), "token")

    for i in range(2):
        stack_step(STACK_STEPS + i)
    torch.cuda.synchronize()
    kgraph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(cap_stream):
        with torch.cuda.graph(kgraph, stream=cap_stream):
            for i in range(STACK_STEPS):
                stack_step(i)
    torch.cuda.synchronize()
    d0.record(stream)
    kgraph.replay()
    d1.record(stream)
    torch.cuda.synchronize()
    stack_us = 1e3 * d0.elapsed_time(d1) / STACK_STEPS
    stack_bytes = STACK_LAYERS * decode_bytes(ss)
    stack_state_mb = STACK_LAYERS * o1.o1_state_bytes(gs) / 1e6
    for st_ in sstates:
        assert o1.o1_state_flags(st_, gs) == 0, "state flags raised"
    del sstates, sscr

    # ---- roofline of the dominant kernel (the window attention)
    pk_, src = peaks()
    names = [o1.o1_stage_name(j) for j in range(nst)]
    near_ms = float(stage_avg[names.index("near")])
    flops = window_flops(sh, ROWS)
    ach = flops / (near_ms * 1e-3) / 1e12
    if tensor_core_window(sh):
        # fp16 tensor cores (same dense rate as bf16); each fp32 product costs
        # three fp16 products (hi.hi + hi.lo + lo.hi), so peak / 3 is this
        # formulation's own ceiling
        peak = pk_["bf16_tflops"]
        traffic = traffic_record("k_near_tc")
        roof = {"kernel": "k_near_tc (window attention, tcgen05 kind::f16, 3-term fp16 split)",
                "bound": "tensor", "achieved": ach, "peak": peak, "unit": "TFLOP/s", "frac": ach / peak,
                "traffic": traffic,
                "peak_source": f"{src} bf16 burst (dense fp16 runs at the bf16 rate)",
                "issued_tensor_tflops": 3 * ach, "frac_of_split_ceiling": 3 * ach / peak,
                "algorithmic_flops_per_launch": flops, "launch_ms": near_ms}
        launches = nst
    else:
        traffic = traffic_record("k_near")
        roof = {"kernel": "k_near (window attention, fp32 CUDA cores)", "bound": "alu", "achieved": ach,
                "peak": FP32_PEAK_TFLOPS, "unit": "TFLOP/s", "frac": ach / FP32_PEAK_TFLOPS, "traffic": traffic,
                "peak_source": "derived: 152 SMs x 128 FP32 lanes x 2 flop x 2070 MHz",
                "algorithmic_flops_per_launch": flops, "launch_ms": near_ms}
        launches = nst - 1   # no panel gather

    value = whole_job_rate(ROWS, args.steps, world, ms_max)
    line = {"metric": METRIC, "value": value, "unit": "rows/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": WORKLOAD, "parallelism": f"replicas x{world} (KV groups and layers are "
                       "independent; no exchange)",
                       "l2": f"inputs larger than L2: {N_SETS} rotating input sets of {set_bytes / 1e6:.0f} MB "
                             f"+ {scratch.numel() / 1e6:.0f} MB scratch",
                       "step": "device copy of the fresh state + o1_chunk_attend(rows=4096)"},
            "roofline": roof,
            "stages_ms": {o1.o1_stage_name(j): float(stage_avg[j]) for j in range(nst)},
            "gpu_launches": launches * args.steps,
            "e2e": {"value": ROWS * args.steps * world / (e2e_ms * 1e-3), "unit": "rows/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "decode": {"metric": "sealed-layer decode us/token", "value": dec_us, "unit": "us/token",
                       "higher_is_better": False,
                       "config": "same layer after an 8192-row prompt; 256 one-row o1_token_attend steps, "
                                 "each evicting one key, captured once in a CUDA graph and replayed",
                       "gpu_launches_per_step": dec_launches,
                       "algorithmic_bytes_per_step": dec_bytes,
                       "achieved_gbs": dec_bytes / (dec_us * 1e-6) / 1e9,
                       "hbm_peak_gbs": pk_["hbm_gbs"],
                       "frac_of_hbm": dec_bytes / (dec_us * 1e-6) / 1e9 / pk_["hbm_gbs"],
                       "note": "the 9.3 MB state stays in L2 across steps"},
            "comparator": {"metric": "exact causal attention rows/s (same prompt, window = 4096, no sinks, "
                                     "no far field)", "value": ROWS / (x_ms * 1e-3), "unit": "rows/s",
                           "ms_per_prompt": x_ms, "sealed_ms_per_prompt": ms_max / args.steps,
                           "algorithmic_tflops": x_flops / (x_ms * 1e-3) / 1e12,
                           "config": "o1_window_attend over the 4096-row prompt from a fresh state, the inputs "
                                     "rotating through the same sets as the prefill steps"},
            "decode_stack": {"metric": "sealed-layer decode us per 24-layer token (stack shape, states larger than "
                                       "L2)", "value": stack_us, "unit": "us/token", "higher_is_better": False,
                             "config": f"{STACK_LAYERS} independent layers G=4 x 4 heads, d=dv=128, 4 sinks, "
                                       f"window 1024, 64 landmarks, each prefilled with {STACK_PREFILL} rows; "
                                       f"{STACK_STEPS} steps through all layers captured once in a CUDA graph",
                             "states_mb": stack_state_mb,
                             "gpu_launches_per_step": 2 * STACK_LAYERS,
                             "algorithmic_bytes_per_step": stack_bytes,
                             "achieved_gbs": stack_bytes / (stack_us * 1e-6) / 1e9,
                             "hbm_peak_gbs": pk_["hbm_gbs"],
                             "frac_of_hbm": stack_bytes / (stack_us * 1e-6) / 1e9 / pk_["hbm_gbs"]},
            "rewind": {"metric": "o1_state_back(1) + one-row o1_spec_commit us/pair", "value": back_us,
                       "unit": "us/pair", "higher_is_better": False,
                       "config": f"{SPEC_CYCLES} pairs on the decode state, captured once in a CUDA graph"},
            "speculative": {"metric": "sealed-layer speculative verify + commit us/cycle", "value": spec_us,
                            "unit": "us/cycle", "higher_is_better": False,
                            "accepted_rows_per_s": SPEC_ACC / (spec_us * 1e-6),
                            "config": f"after the decode steps: {SPEC_DRAFT}-row drafts through "
                                      f"o1_chunk_attend_spec, {SPEC_ACC} rows of each through o1_spec_commit; "
                                      f"{SPEC_CYCLES} cycles captured once in a CUDA graph and replayed",
                            "gpu_launches_per_cycle": nst - 1 + 4},
            "peaks": {"source": src, **{k2: pk_[k2] for k2 in ("hbm_gbs", "bf16_tflops") if k2 in pk_}},
            "clocks": clk.summary()}
    if rank == 0 and world == 1:
        rate, dt, cores = oracle_prompt_rate(ROWS, SHAPE.groups)
        line["cpu_baseline"] = {"value": rate, "unit": "rows/s", "cores": cores, "kind": "oracle",
                                "sample": f"the whole 4096-row prompt once ({dt:.1f} s)"}
    if rank == 0:
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        reference_arm(args, rank)
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    our_arm(args, rank, world, local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
