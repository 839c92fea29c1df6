"""Writes tests/golden/page_case_*.txt from the oracle alone.

The pages print no expected values. These fixtures pin the oracle's output on
the pages' own small test scenarios (see tests/scenarios.py) against later
changes of the oracle itself; the GPU path is compared with the live oracle.
Run from the repository root: python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))
sys.path.insert(0, os.path.dirname(HERE))

import oracle  # noqa: E402
import scenarios  # noqa: E402


def run_case(idx):
    shape, c, prompt, chunks = scenarios.page_case(*scenarios.PAGE_CASES[idx])
    g = oracle.Geom(shape.groups, shape.heads_per_group, shape.d, shape.dv, shape.sinks, shape.window,
                    shape.landmarks, rope_base=shape.rope_base)
    lay = oracle.OracleLayer(g, c.sink_k, c.sink_v, c.k_tilde, c.q_tilde, c.mu,
                             group_windows=shape.group_windows)
    lay.rows(*prompt)
    return [lay.rows(*ch) for ch in chunks]


def main():
    for idx in (0, 1):
        outs = run_case(idx)
        path = os.path.join(HERE, f"page_case_{idx}.txt")
        with open(path, "w") as f:
            f.write(f"# oracle output of page scenario {scenarios.PAGE_CASES[idx]} (d, m, w, sink, hpg, t, w2, chunks)\n")
            f.write("# from 'cortiq-engine 0.8.51 src/gpu_wgpu/o1_batch.rs' test o1_batch_matches_serial_steps;\n")
            f.write("# written by tests/golden/make_golden.py (oracle only). Columns: chunk row head out[0..dv)\n")
            for ci, o in enumerate(outs):
                for r in range(o.shape[0]):
                    for h in range(o.shape[1]):
                        f.write(f"{ci} {r} {h} " + " ".join(f"{x:.15e}" for x in o[r, h]) + "\n")
        print("wrote", path)


if __name__ == "__main__":
    main()
