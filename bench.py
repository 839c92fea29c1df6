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
L2 (`decode_stack`), both against HBM; the same prompt as 64-row calls
(`prefill_chunked`); a 32768-row prompt with group windows 1024 / 2048
(`long_prompt`); the 24-layer stack's prefill in 64-row chunks
(`stack_prefill`); exact causal attention over the same prompt
(`comparator`); speculative verify + commit cycles (`speculative`); ring
rewinds (`rewind`).

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


def device_rows(torch, shape: synth.Shape, seed: int, rows: int, dev, gate: bool = True):
    """Seeded N(0,1) rows made on the device with torch's generator (one
    stream per (seed, tensor)), for workloads too large to draw through the
    host generator within a benchmark run. Untimed, and never compared with
    the oracle (the parity tests draw their inputs from synth)."""
    g = torch.Generator(device=dev)

    def draw(tensor, shp):
        g.manual_seed(seed * 16 + tensor)
        return torch.randn(shp, generator=g, device=dev, dtype=torch.float32)
    q = draw(synth.Q, (rows, shape.nh, shape.d))
    k = draw(synth.K, (rows, shape.groups, shape.d))
    v = draw(synth.V, (rows, shape.groups, shape.dv))
    gt = draw(synth.GATE, (rows, shape.nh, shape.dv)) if gate else None
    return q, k, v, gt


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


def oracle_one_thread_rates():
    """The oracle on one thread: the tiny workload in full (16 + 64 rows) and
    the first 1024 rows of the Qwen-layer prompt."""
    import oracle
    out = {}
    for name, sh, seed, rows in (("tiny", synth.TINY, 0, 80), ("qwen_layer_1024_rows", SHAPE, SEED, 1024)):
        c = synth.layer_constants(sh, seed)
        g = oracle.Geom(sh.groups, sh.heads_per_group, sh.d, sh.dv, sh.sinks, sh.window, sh.landmarks,
                        rope_base=sh.rope_base)
        lay = oracle.OracleLayer(g, c.sink_k, c.sink_v, c.k_tilde, c.q_tilde, c.mu)
        q, k, v, gt = synth.layer_rows(sh, seed, 0, rows)
        t0 = time.perf_counter()
        lay.rows(q, k, v, gt, threads=1)
        out[name] = {"rows": rows, "seconds": time.perf_counter() - t0,
                     "rows_per_s": rows / (time.perf_counter() - t0)}
    return out


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

    # ---- end to end: host buffers in, host output back, through the C ABI.
    # As a serving loop runs it: two device input sets; while step i
    # computes, step i+1's inputs go up on one copy stream and step i-1's
    # output comes down on another. Every step still copies its own inputs
    # from pinned host memory and reads its output back inside the timed
    # region; events order each buffer's reuse.
    host_outs = [torch.empty((ROWS, sh.nh, sh.dv), dtype=torch.float32).pin_memory() for _ in range(2)]
    bufs = [sets[0], sets[1 % N_SETS]]
    up_st, down_st = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]     # set b's inputs are on the device
    ev_done = [torch.cuda.Event() for _ in range(2)]   # set b's step has computed (inputs free, output ready)
    ev_out = [torch.cuda.Event() for _ in range(2)]    # set b's output is on the host (buffer free)
    for b in range(2):
        ev_done[b].record(stream)
        ev_out[b].record(stream)

    def e2e_upload(i):
        b = i % 2
        up_st.wait_event(ev_done[b])
        with torch.cuda.stream(up_st):
            for name, h in (("q", hq), ("k", hk), ("v", hv), ("g", hg)):
                bufs[b][name].copy_(h, non_blocking=True)
        ev_in[b].record(up_st)

    def e2e_compute(i):
        b = i % 2
        stream.wait_event(ev_in[b])
        stream.wait_event(ev_out[b])
        bufs[b]["state"].copy_(pristine, non_blocking=True)
        o1.check(o1.o1_chunk_attend(bufs[b]["state"], g, scratch, bufs[b]["q"], bufs[b]["k"], bufs[b]["v"],
                                    bufs[b]["g"], ROWS, bufs[b]["out"]), "chunk")
        ev_done[b].record(stream)
        down_st.wait_event(ev_done[b])
        with torch.cuda.stream(down_st):
            host_outs[b].copy_(bufs[b]["out"], non_blocking=True)
        ev_out[b].record(down_st)

    def e2e_run(n):
        for st_ in (up_st, down_st):   # nothing of the run starts before the start event
            st_.wait_stream(stream)
        e2e_upload(0)
        for i in range(n):
            if i + 1 < n:
                e2e_upload(i + 1)
            e2e_compute(i)
        stream.wait_event(ev_out[(n - 1) % 2])
        stream.wait_event(ev_out[n % 2])

    e2e_run(max(1, args.warmup))
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_run(args.steps)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hg))
    d2h = host_outs[0].numel() * 4

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
    dec_launches = 1

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
    pout = torch.empty((STACK_PREFILL, ss.nh, ss.dv), dtype=torch.float32, device=dev)
    sstates, st_rows = [], []
    for layer in range(STACK_LAYERS):
        cl = synth.layer_constants(ss, 1000 + layer)
        cst = [up(cl.sink_k), up(cl.sink_v), up(cl.k_tilde), up(cl.q_tilde), up(cl.mu)]
        st_ = torch.empty(o1.o1_state_bytes(gs), dtype=torch.uint8, device=dev)
        o1.check(o1.o1_state_init(st_, gs, None, *cst, 0), "init")
        rq, rk, rv, rg = device_rows(torch, ss, 1000 + layer, STACK_PREFILL + STACK_STEPS + 2, dev)
        o1.check(o1.o1_chunk_attend(st_, gs, sscr, rq[:STACK_PREFILL], rk[:STACK_PREFILL], rv[:STACK_PREFILL],
                                    rg[:STACK_PREFILL], STACK_PREFILL, pout), "prefill")
        sstates.append(st_)
        st_rows.append((rq[STACK_PREFILL:], rk[STACK_PREFILL:], rv[STACK_PREFILL:], rg[STACK_PREFILL:]))
    del pout
    souts = [torch.empty((ss.nh, ss.dv), dtype=torch.float32, device=dev) for _ in range(STACK_LAYERS)]

    def stack_step(i):
        for st_, (sq_, sk_, sv_, sg_), so_ in zip(sstates, st_rows, souts):
            o1.check(o1.o1_token_attend(st_, gs, sscr, sq_[i], sk_[i], sv_[i], sg_[i], so_), "token")

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

    pk_, src = peaks()
    steps_big = max(2, min(args.steps, 5))

    def graph_of(fn):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.stream(cap_stream):
            with torch.cuda.graph(gr, stream=cap_stream):
                fn()
        torch.cuda.synchronize()
        return gr

    def timed_replays(graphs, restore, n):
        """Mean ms of a graph replay; restore() runs before each, untimed."""
        tot = 0.0
        for i in range(n):
            restore(i)
            torch.cuda.synchronize()
            d0.record(stream)
            graphs[i % len(graphs)].replay()
            d1.record(stream)
            torch.cuda.synchronize()
            tot += d0.elapsed_time(d1)
        return tot / n

    # ---- the same 4096-row prompt as 64 calls of 64 rows (the pages' model
    # calls the batch kernels once per 64-row chunk), each input set's 64
    # calls captured once in a CUDA graph; the fresh state restored before
    # each replay, outside the timed region
    cscratch = torch.empty(o1.o1_scratch_bytes(g, 64), dtype=torch.uint8, device=dev)
    cstate = torch.empty(sbytes, dtype=torch.uint8, device=dev)

    def chunk_calls(s_):
        def run():
            for r0 in range(0, ROWS, 64):
                o1.check(o1.o1_chunk_attend(cstate, g, cscratch, s_["q"][r0:r0 + 64], s_["k"][r0:r0 + 64],
                                            s_["v"][r0:r0 + 64], s_["g"][r0:r0 + 64], 64, s_["out"][r0:r0 + 64]),
                         "chunk")
        return run
    cstate.copy_(pristine)
    chunk_calls(sets[0])()   # first calls on this thread: the library's second stream, attributes
    cgraphs = [graph_of(chunk_calls(s_)) for s_ in sets]
    c64_ms = timed_replays(cgraphs, lambda i: cstate.copy_(pristine), max(3, args.steps))
    c64_flops = window_flops(sh, ROWS)
    del cgraphs, cscratch, cstate

    # ---- the long prompt: 32768 rows, group windows 1024 and 2048, one call
    lsh = synth.QWEN_LONG
    gl = o1.geom(lsh.groups, lsh.heads_per_group, lsh.d, lsh.dv, lsh.sinks, lsh.window, lsh.landmarks,
                 rope_base=lsh.rope_base)
    LROWS = 32768
    lc = synth.layer_constants(lsh, 3)
    lconsts = [up(lc.sink_k), up(lc.sink_v), up(lc.k_tilde), up(lc.q_tilde), up(lc.mu)]
    lpristine = torch.empty(o1.o1_state_bytes(gl), dtype=torch.uint8, device=dev)
    o1.check(o1.o1_state_init(lpristine, gl, lsh.group_windows, *lconsts, 0), "init")
    lstate = torch.empty_like(lpristine)
    lscratch = torch.empty(o1.o1_scratch_bytes(gl, LROWS), dtype=torch.uint8, device=dev)
    lq, lk, lv, lg = device_rows(torch, lsh, 3, LROWS, dev)
    lout = torch.empty((LROWS, lsh.nh, lsh.dv), dtype=torch.float32, device=dev)
    lgraph = graph_of(lambda: o1.check(o1.o1_chunk_attend(lstate, gl, lscratch, lq, lk, lv, lg, LROWS, lout),
                                       "long"))
    long_ms = timed_replays([lgraph], lambda i: lstate.copy_(lpristine), steps_big)
    long_flops = window_flops(lsh, LROWS)
    assert o1.o1_state_flags(lstate, gl) == 0, "state flags raised"
    del lgraph, lscratch, lq, lk, lv, lg, lout, lstate, lpristine

    # ---- the 24-layer stack's prefill, chunk-major as a model runs it: for
    # each 64-row chunk every layer in turn. Each layer is first brought to
    # its steady state (the ring full: 1088 rows in one untimed call); then
    # STACK_CHUNKS chunks go through all layers, captured once in a CUDA
    # graph, the states restored before each replay outside the timed region.
    STACK_CHUNKS = 16
    ss = synth.STACK_LAYER
    gs = o1.geom(ss.groups, ss.heads_per_group, ss.d, ss.dv, ss.sinks, ss.window, ss.landmarks,
                 rope_base=ss.rope_base)
    sbytes_s = o1.o1_state_bytes(gs)
    pscr = torch.empty(o1.o1_scratch_bytes(gs, 1088), dtype=torch.uint8, device=dev)
    cscr = torch.empty(o1.o1_scratch_bytes(gs, 64), dtype=torch.uint8, device=dev)
    warm_states, live_states, layer_rows = [], [], []
    for layer in range(STACK_LAYERS):
        cl = synth.layer_constants(ss, 1000 + layer)
        cst = [up(cl.sink_k), up(cl.sink_v), up(cl.k_tilde), up(cl.q_tilde), up(cl.mu)]
        st_ = torch.empty(sbytes_s, dtype=torch.uint8, device=dev)
        o1.check(o1.o1_state_init(st_, gs, None, *cst, 0), "init")
        rq, rk, rv, rg = device_rows(torch, ss, 1000 + layer, 1088 + 64 * STACK_CHUNKS, dev)
        pout = torch.empty((1088, ss.nh, ss.dv), dtype=torch.float32, device=dev)
        o1.check(o1.o1_chunk_attend(st_, gs, pscr, rq[:1088], rk[:1088], rv[:1088], rg[:1088], 1088, pout),
                 "prefill")
        warm_states.append(st_)
        live_states.append(torch.empty_like(st_))
        layer_rows.append((rq[1088:], rk[1088:], rv[1088:], rg[1088:],
                           torch.empty((64 * STACK_CHUNKS, ss.nh, ss.dv), dtype=torch.float32, device=dev)))
    del pscr, pout

    def restore_stack(i):
        for a_, b_ in zip(live_states, warm_states):
            a_.copy_(b_)

    def stack_chunks():
        for c in range(STACK_CHUNKS):
            r0 = 64 * c
            for layer in range(STACK_LAYERS):
                q_, k_, v_, g_, o_ = layer_rows[layer]
                o1.check(o1.o1_chunk_attend(live_states[layer], gs, cscr, q_[r0:r0 + 64], k_[r0:r0 + 64],
                                            v_[r0:r0 + 64], g_[r0:r0 + 64], 64, o_[r0:r0 + 64]), "chunk")
    restore_stack(0)
    sgraph_p = graph_of(stack_chunks)
    stack_ms = timed_replays([sgraph_p], restore_stack, steps_big)
    stack_rows = 64 * STACK_CHUNKS
    stack_flops = STACK_LAYERS * window_flops(ss, stack_rows, len0=ss.window)
    for st_ in live_states:
        assert o1.o1_state_flags(st_, gs) == 0, "state flags raised"
    del sgraph_p, warm_states, live_states, layer_rows, cscr

    # ---- roofline of the dominant kernel (the window attention)
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
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "note": "pinned host buffers; two device input sets, the next step's upload and the "
                            "previous step's download on their own streams beside the current step"},
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
                                       f"window 1024, 64 landmarks (per-layer constants and rows from seeds "
                                       f"1000 + layer, rows drawn on the device), each prefilled with "
                                       f"{STACK_PREFILL} rows; {STACK_STEPS} steps through all layers captured once "
                                       f"in a CUDA graph",
                             "states_mb": stack_state_mb,
                             "gpu_launches_per_step": STACK_LAYERS,
                             "algorithmic_bytes_per_step": stack_bytes,
                             "achieved_gbs": stack_bytes / (stack_us * 1e-6) / 1e9,
                             "hbm_peak_gbs": pk_["hbm_gbs"],
                             "frac_of_hbm": stack_bytes / (stack_us * 1e-6) / 1e9 / pk_["hbm_gbs"]},
            "prefill_chunked": {"metric": "sealed-layer prefill rows/s, the 4096-row prompt as 64 calls of 64 rows",
                                "value": ROWS / (c64_ms * 1e-3), "unit": "rows/s", "ms_per_prompt": c64_ms,
                                "algorithmic_tflops": c64_flops / (c64_ms * 1e-3) / 1e12,
                                "frac_of_bf16_peak": c64_flops / (c64_ms * 1e-3) / 1e12 / pk_["bf16_tflops"],
                                "config": "same layer and inputs as the prefill steps; 64 o1_chunk_attend calls of "
                                          "64 rows each, per input set captured once in a CUDA graph; the fresh "
                                          "state restored before each replay, untimed"},
            "long_prompt": {"metric": "sealed-layer prefill rows/s, 32768-row prompt, group windows 1024 / 2048",
                            "value": LROWS / (long_ms * 1e-3), "unit": "rows/s", "ms_per_prompt": long_ms,
                            "algorithmic_tflops": long_flops / (long_ms * 1e-3) / 1e12,
                            "frac_of_bf16_peak": long_flops / (long_ms * 1e-3) / 1e12 / pk_["bf16_tflops"],
                            "config": "Qwen3.5-0.8B-shaped layer with group windows 1024 and 2048 (meta slot 3), "
                                      "one o1_chunk_attend of 32768 rows from a fresh state (inputs drawn on the "
                                      "device, seed 3); state restored before each run, untimed"},
            "stack_prefill": {"metric": "24-layer stack prefill rows/s (64-row chunks, chunk-major, steady state)",
                              "value": stack_rows / (stack_ms * 1e-3), "unit": "rows/s",
                              "ms_per_chunk_through_24_layers": stack_ms / STACK_CHUNKS,
                              "projected_65536_row_prompt_s": 65536 / (stack_rows / (stack_ms * 1e-3)),
                              "algorithmic_tflops": stack_flops / (stack_ms * 1e-3) / 1e12,
                              "frac_of_bf16_peak": stack_flops / (stack_ms * 1e-3) / 1e12 / pk_["bf16_tflops"],
                              "config": f"{STACK_LAYERS} layers G=4 x 4 heads, d=dv=128, 4 sinks, window 1024, 64 "
                                        f"landmarks (per-layer constants from seeds 1000 + layer, per-layer rows drawn "
                                        f"on the device); each layer brought to its full ring by an untimed "
                                        f"1088-row call, then {STACK_CHUNKS} chunks of 64 rows through every layer "
                                        f"in turn ({STACK_CHUNKS * STACK_LAYERS} calls) in one CUDA graph; states "
                                        f"restored before each replay, untimed. A stated subset of the 65536-row "
                                        f"prompt: its rows past the first window cost the same per chunk"},
            "rewind": {"metric": "o1_state_back(1) + one-row o1_spec_commit us/pair", "value": back_us,
                       "unit": "us/pair", "higher_is_better": False,
                       "config": f"{SPEC_CYCLES} pairs on the decode state, captured once in a CUDA graph",
                       "gpu_launches_per_pair": 2},
            "speculative": {"metric": "sealed-layer speculative verify + commit us/cycle", "value": spec_us,
                            "unit": "us/cycle", "higher_is_better": False,
                            "accepted_rows_per_s": SPEC_ACC / (spec_us * 1e-6),
                            "config": f"after the decode steps: {SPEC_DRAFT}-row drafts through "
                                      f"o1_chunk_attend_spec, {SPEC_ACC} rows of each through o1_spec_commit; "
                                      f"{SPEC_CYCLES} cycles captured once in a CUDA graph and replayed",
                            # verify: rotation, short far kernel, key-slice window kernel and
                            # its slice merge, merge; commit: short far kernel, ring push
                            "gpu_launches_per_cycle": 7},
            "peaks": {"source": src, **{k2: pk_[k2] for k2 in ("hbm_gbs", "bf16_tflops") if k2 in pk_}},
            "clocks": clk.summary()}
    if rank == 0 and world == 1:
        rate, dt, cores = oracle_prompt_rate(ROWS, SHAPE.groups)
        line["cpu_baseline"] = {"value": rate, "unit": "rows/s", "cores": cores, "kind": "oracle",
                                "sample": f"the whole 4096-row prompt once ({dt:.1f} s), KV groups on "
                                          f"{cores} threads (rows are serial)",
                                "host_cores": os.cpu_count(), "threads_used": cores,
                                "one_thread": oracle_one_thread_rates()}
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
