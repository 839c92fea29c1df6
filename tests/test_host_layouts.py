"""The device memory maps on the host, over a grid of geometries (no GPU):
the state's and a call's scratch parts start on 256 bytes and follow one
another without overlap; the scratch holds the key-split window partials of
every pass it can run; the one-row path's far chunks and near slices cover
every landmark and every near key, none of them empty."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

DRIVER = r"""
#include <cstdio>
#include <cstring>
#include "o1_common.cuh"

static int failures = 0;
#define CHECK(c, ...) do { if (!(c)) { if (failures < 20) { printf("FAIL %s: ", #c); printf(__VA_ARGS__); printf("\n"); } ++failures; } } while (0)

static void contiguous(const char *what, const size_t *off, int n, size_t total, const o1_geom &g) {
    CHECK(off[0] == 0, "%s starts at %zu", what, off[0]);
    for (int i = 0; i < n; ++i) {
        CHECK(off[i] % 256 == 0, "%s part %d at %zu (G %d d %d dv %d)", what, i, off[i], g.groups, g.d, g.dv);
        const size_t next = i + 1 < n ? off[i + 1] : total;
        CHECK(next >= off[i], "%s part %d overlaps", what, i);
    }
}

int main() {
    const int Gs[] = {1, 2, 4, 16}, hpgs[] = {1, 2, 4, 16}, ds[] = {8, 64, 128, 256}, dvs[] = {4, 64, 128, 256};
    const int nss[] = {0, 4, 64}, ws[] = {1, 16, 512, 2048, 65536}, ms[] = {1, 8, 32, 64};
    const int caps[] = {1, 2, 64, 300, 4096};
    long geoms = 0, tok_over = 0;
    for (int G : Gs) for (int hpg : hpgs) for (int d : ds) for (int dv : dvs) for (int ns : nss) for (int w : ws)
    for (int m : ms) {
        o1_geom g;
        memset(&g, 0, sizeof(g));
        g.groups = G; g.heads_per_group = hpg; g.d = d; g.dv = dv; g.sinks = ns; g.window = w; g.landmarks = m;
        g.scale = 1.f;
        ++geoms;
        const size_t nh = (size_t)G * hpg;
        // the state
        const O1Layout L = o1_layout(g);
        const size_t so[] = {L.hdr, L.meta, L.ring_k, L.ring_v, L.sink_k, L.sink_v, L.kt, L.qt, L.mu, L.M, L.Z,
                             L.Zlo, L.T, L.tick};
        contiguous("state", so, 14, L.total, g);
        CHECK(L.ring_v - L.ring_k >= (size_t)G * w * d * 4, "ring_k size");
        CHECK(L.T + nh * m * dv * 4 <= L.tick, "T size");
        CHECK(L.total - L.tick >= (nh + G + 1) * 4, "arrival counters");
        // a call's scratch
        for (int cap : caps) {
            const O1Scratch S = o1_scratch_layout(g, cap);
            const size_t co[] = {S.qr, S.kr, S.E, S.P, S.Fb, S.Tp, S.fh, S.sh, S.sn, S.Xk, S.XvT, S.Qs, S.Sp, S.Wp};
            contiguous("scratch", co, 14, S.total, g);
            CHECK(S.ldc % 4 == 0 && S.ldc >= cap, "ldc %d cap %d", S.ldc, cap);
            CHECK(S.Fb + ((size_t)O1_FB_PLANES * S.nsub + 3) * nh * m * 4 <= S.Tp, "Fb with its entering planes");
            if (cap >= 2)
                CHECK(S.Wp - S.Sp >= (size_t)G * O1_SMALL_NS * O1_SMALL_NQ * (dv + 2) * 4, "Sp size");
            // every pass of R <= cap rows that splits its window keys S ways
            // finds (S - 1) R rows of partials and headers
            const int Rs[] = {2, 3, 64, 127, 128, 129, 255, 256, 300, 1000, 4096};
            for (int R : Rs) {
                if (R > cap) continue;
                const int Sw = o1_wsplit(g, R);
                CHECK(Sw >= 1, "wsplit %d", Sw);
                if (Sw > 1)
                    CHECK(S.total - S.Wp >= (size_t)(Sw - 1) * R * nh * (dv + 4) * 4,
                          "Wp for R %d S %d (G %d hpg %d w %d)", R, Sw, G, hpg, w);
            }
        }
        // the one-row path
        const O1TokScratch T = o1_tok_layout(g);
        const long nnear = (long)ns + w;
        CHECK(T.MB >= 1 && T.MB <= O1_TOK_MB_MAX, "MB %d", T.MB);
        CHECK((long)T.NF * T.MB >= m && (long)(T.NF - 1) * T.MB < m, "far chunks NF %d MB %d m %d", T.NF, T.MB, m);
        CHECK(T.KC % 8 == 0 && T.KC >= 8 && T.KC <= 256, "KC %d", T.KC);
        CHECK((long)T.NC * T.KC >= nnear && (long)(T.NC - 1) * T.KC < nnear, "near slices NC %d KC %d n %ld",
              T.NC, T.KC, nnear);
        CHECK(T.smem % 4 == 0, "smem %zu", T.smem);
        const size_t to[] = {T.part, T.pml, T.farp, T.kcur};
        contiguous("one-row scratch", to, 4, T.total, g);
        CHECK(T.pml - T.part >= (size_t)G * T.NC * hpg * dv * 4, "part size");
        CHECK(T.kcur - T.farp >= nh * T.NF * (4 + dv) * 4, "farp size");
        if (T.smem > 227 * 1024) ++tok_over;   // refused at launch (invalid configuration), not run
        CHECK(o1_scratch_need(g, 64) >= T.total && o1_scratch_need(g, 64) >= o1_scratch_layout(g, 64).total,
              "scratch_need");
    }
    printf("geometries %ld one-row layouts above 227 KB %ld failures %d\n", geoms, tok_over, failures);
    return failures ? 1 : 0;
}
"""


def test_state_scratch_and_one_row_layouts(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    src = tmp_path / "host_layouts.cu"
    src.write_text(DRIVER)
    exe = tmp_path / "host_layouts"
    csrc = os.path.join(ROOT, "sliding_window_landmark_gb300", "csrc")
    subprocess.run([nvcc, "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a", "-I", csrc,
                    "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True, capture_output=True, timeout=300)
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert run.returncode == 0, run.stdout + run.stderr
    assert "failures 0" in run.stdout, run.stdout
