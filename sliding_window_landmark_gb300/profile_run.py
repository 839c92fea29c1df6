"""A fixed launch sequence for profilers: one sealed layer, `--calls` chunk
calls of `--rows` rows each from a fresh state (the state restored between
calls), or `--tokens` one-row calls after a prompt of `--rows` rows.

  python -m sliding_window_landmark_gb300.profile_run --shape qwen --rows 4096 --calls 3
  python -m sliding_window_landmark_gb300.profile_run --shape qwen --rows 8192 --tokens 16
  python -m sliding_window_landmark_gb300.profile_run --shape qwen --rows 8192 --spec 8,5 --cycles 3

Launches per chunk call: rope, then far_block, far_tscan, side_readout on a
second stream beside [gather_tc], near, then merge, commit;
per one-row call: k_tok (one launch); per speculative cycle (`--spec
DRAFT,ACCEPTED`): the attend-only pass of the draft (no commit kernel; for a
draft of at most 16 rows the key-slice window kernels beside the short far
kernel), then the commit pass of the accepted rows (rope, the short far
kernel or far_block + far_tscan, commit). The library must already be built.
"""
from __future__ import annotations

import argparse

import numpy as np
import torch

from . import o1, synth

SHAPES = {"tiny": synth.TINY, "qwen": synth.QWEN_LAYER, "qwen_long": synth.QWEN_LONG,
          "stack": synth.STACK_LAYER}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--shape", choices=sorted(SHAPES), default="qwen")
    ap.add_argument("--rows", type=int, default=4096)
    ap.add_argument("--calls", type=int, default=3)
    ap.add_argument("--tokens", type=int, default=0)
    ap.add_argument("--seed", type=int, default=1)
    ap.add_argument("--spec", default="", help="DRAFT,ACCEPTED rows of speculative cycles after the prompt")
    ap.add_argument("--cycles", type=int, default=3)
    args = ap.parse_args()
    sh = SHAPES[args.shape]
    dev = torch.device("cuda")
    g = o1.geom(sh.groups, sh.heads_per_group, sh.d, sh.dv, sh.sinks, sh.window, sh.landmarks,
                rope_base=sh.rope_base)
    c = synth.layer_constants(sh, args.seed)
    up = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev)
    consts = [up(c.sink_k), up(c.sink_v), up(c.k_tilde), up(c.q_tilde), up(c.mu)]
    state = torch.empty(o1.o1_state_bytes(g), dtype=torch.uint8, device=dev)
    o1.check(o1.o1_state_init(state, g, sh.group_windows, *consts, 0), "init")
    fresh = state.clone()
    scratch = torch.empty(o1.o1_scratch_bytes(g, args.rows), dtype=torch.uint8, device=dev)
    q, k, v, gt = (up(x) for x in synth.layer_rows(sh, args.seed, 0, args.rows))
    out = torch.empty((args.rows, sh.nh, sh.dv), dtype=torch.float32, device=dev)
    if args.spec:
        nd, na = (int(x) for x in args.spec.split(","))
        o1.check(o1.o1_chunk_attend(state, g, scratch, q, k, v, gt, args.rows, out), "prompt")
        sq, sk, sv, sg = (up(x) for x in synth.layer_rows(sh, args.seed, args.rows, nd * args.cycles))
        sout = torch.empty((nd, sh.nh, sh.dv), dtype=torch.float32, device=dev)
        for i in range(args.cycles):
            a, b = i * nd, (i + 1) * nd
            o1.check(o1.o1_chunk_attend_spec(state, g, scratch, sq[a:b], sk[a:b], sv[a:b], sg[a:b], nd, sout), "spec")
            o1.check(o1.o1_spec_commit(state, g, scratch, sk[a:a + na], sv[a:a + na], na), "commit")
        out = sout
    elif args.tokens:
        o1.check(o1.o1_chunk_attend(state, g, scratch, q, k, v, gt, args.rows, out), "prompt")
        tq, tk, tv, tg = (up(x) for x in synth.layer_rows(sh, args.seed, args.rows, args.tokens))
        tout = torch.empty((args.tokens, sh.nh, sh.dv), dtype=torch.float32, device=dev)
        for i in range(args.tokens):
            o1.check(o1.o1_token_attend(state, g, scratch, tq[i], tk[i], tv[i], tg[i], tout[i]), "token")
    else:
        for _ in range(args.calls):
            state.copy_(fresh)
            o1.check(o1.o1_chunk_attend(state, g, scratch, q, k, v, gt, args.rows, out), "chunk")
    torch.cuda.synchronize()
    assert o1.o1_state_flags(state, g) == 0, "state flags raised"
    assert torch.isfinite(out).all().item()
    print("done", args.shape, args.rows, args.calls, args.tokens)


if __name__ == "__main__":
    main()
