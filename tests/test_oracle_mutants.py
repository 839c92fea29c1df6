"""The oracle's pins catch plausible mistakes.

Each case plants one mistake in a private copy of the oracle's C source
(dropped term, wrong sign, wrong index, transposed operand, skipped branch),
compiles it on the CPU and runs the pins against it: at least one pin must
fail. The unmodified source must pass them all.
"""
import os
import subprocess

import numpy as np
import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "o1_oracle.c")

# (name, text in the oracle, its planted replacement)
MUTANTS = [
    ("far rescale dropped", "double rho = (Mn == Mo) ? 1.0 : exp(Mo - Mn);", "double rho = 1.0;"),
    ("far mass term constant", "st->Z[gh * m + b] = st->Z[gh * m + b] * rho + e;",
     "st->Z[gh * m + b] = st->Z[gh * m + b] * rho + 1.0;"),
    ("far logit unscaled", "double l = scale * oo_dot(qtb, ke, d);", "double l = oo_dot(qtb, ke, d);"),
    ("push slot off by one", "int slot = (head + len) % wg;", "int slot = (head + len + 1) % wg;"),
    ("head not advanced", "if (len == wg) head = (head + 1) % wg;", "if (len == wg) head = head;"),
    ("mu transposed", "acc += exp(f[a] - F) * mu[(size_t)a * m + b];",
     "acc += exp(f[a] - F) * mu[(size_t)b * m + a];"),
    ("sign gate ignored", "if (D >= 0.0) have = 1;", "have = 1;"),
    ("rectifier always on", "if (g->rect && acc < 0.0) acc = 0.0;", "if (acc < 0.0) acc = 0.0;"),
    ("far numerator dropped", "for (int t = 0; t < dv; t++) num[t] += gain[b] * Tb[t];", "(void)Tb;"),
    ("rotation sign", "out[j + half] = b * cs[j] + a * sn[j];", "out[j + half] = b * cs[j] - a * sn[j];"),
    ("rotation frequency", "-2.0 * (double)j / (double)d", "-1.0 * (double)j / (double)d"),
    ("adjacent pairing", "double a = (double)x[j], b = (double)x[j + half];",
     "double a = (double)x[2 * j], b = (double)x[2 * j + 1];"),
    ("window read from wrong slot", "int slot = (head + x) % wg;", "int slot = (head + x + 1) % wg;"),
    ("gate sign", "y = y / (1.0 + exp(-gl));", "y = y / (1.0 + exp(gl));"),
    ("attend before far insert", "if (len == wg) {\n            const double *ke", "if (0) {\n            const double *ke"),
    ("rewind steps the head forward", "mt[1] = (mt[1] + wg - 1) % wg;", "mt[1] = (mt[1] + 1) % wg;"),
    ("rewind keeps the eviction count", "mt[2] -= 1;", "mt[2] -= 0;"),
    ("rewind leaves the position", "*st->pos -= rows;", "*st->pos -= 0;"),
    ("far readout uses landmark keys unscaled", "f[a] = scale * oo_dot(qr, kt + (size_t)a * d, d);",
     "f[a] = oo_dot(qr, kt + (size_t)a * d, d);"),
    ("denominator floor dropped", "if (den < 1e-30) den = 1e-30;", "(void)0;"),
    ("floor taken before the far mass is added", "if (den < 1e-30) den = 1e-30;",
     "den = (den - D < 1e-30 ? 1e-30 : den - D) + D;"),
]


def _pin_calls():
    calls = [pins.test_rope_worked_values, pins.test_rope_invariants,
             pins.test_unit_kernel_closed_form, pins.test_far_state_recomputation_and_monotone_max,
             pins.test_meta_closed_form_and_ring_slots, pins.test_position_shift_invariance,
             pins.test_forced_far_branches, pins.test_meta_rewind_closed_form,
             pins.test_rewind_then_repush_reproduces_rows]
    calls += [lambda lib, rb=rb: pins.test_no_eviction_is_exact_softmax(rb, lib=lib) for rb in (1e6, 0.0)]
    calls += [lambda lib, c=c: pins.test_brute_force_far_algebra(c, lib=lib) for c in pins.BRUTE_CASES]
    calls += [lambda lib, mv=mv: pins.test_denominator_floor(mv, lib=lib) for mv in pins.FLOOR_CASES]
    return calls


def _failures(lib):
    n = 0
    for call in _pin_calls():
        try:
            with np.errstate(all="ignore"):
                call(lib=lib)
        except AssertionError:
            n += 1
    return n


def _build(tmp_path, text):
    src = tmp_path / "mut.c"
    src.write_text(text)
    so = tmp_path / "libmut.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                           str(src), "-o", str(so), "-lm", "-lpthread"])
    return oracle.load_library(str(so))


def test_unmodified_oracle_passes_all_pins(tmp_path):
    assert _failures(_build(tmp_path, open(SRC).read())) == 0


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(tmp_path, name, old, new):
    text = open(SRC).read()
    assert text.count(old) == 1, f"mutation site not unique: {name}"
    assert _failures(_build(tmp_path, text.replace(old, new))) > 0, f"pins missed: {name}"
