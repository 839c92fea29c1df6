"""The short far kernel's shared-memory layout and thread split, checked on
the host over a grid of geometries (no GPU): every part starts on 16 bytes
and follows the previous one without overlap, the value columns are split
over CTAs as the launcher expects, the column threads of the value-sum step
cover every column, and their reads of T hit distinct banks."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

DRIVER = r"""
#include <cstdio>
#include <cstring>
#include <set>
#include <map>
#include "o1_common.cuh"

static int failures = 0;
#define CHECK(c, ...) do { if (!(c)) { if (failures < 20) { printf("FAIL %s: ", #c); printf(__VA_ARGS__); printf("\n"); } ++failures; } } while (0)

int main() {
    const int ds[] = {8, 16, 64, 72, 128, 256}, dvs_[] = {4, 12, 16, 20, 64, 96, 128, 256};
    const int ms[] = {1, 3, 8, 32, 64}, nss[] = {0, 1, 4, 64}, Rs[] = {1, 2, 5, 8, 16};
    const int nhs[] = {1, 2, 8, 16, 37, 74, 148, 1024};
    long cases = 0;
    size_t max_bytes = 0;
    for (int d : ds) for (int dv : dvs_) for (int m : ms) for (int ns : nss) for (int R : Rs) for (int nh : nhs) {
        O1Args a;
        memset(&a, 0, sizeof(a));
        a.d = d; a.dv = dv; a.m = m; a.ns = ns; a.R = R; a.nh = nh;
        ++cases;
        const int cs = short_col_splits(a);
        CHECK(cs == 1 || cs == 2 || cs == 4, "cs %d", cs);
        CHECK(cs == 1 || (dv % (4 * cs) == 0 && nh * cs <= 148), "cs %d dv %d nh %d", cs, dv, nh);
        const ShortLayout L = short_layout(a);
        CHECK(L.dvs * cs == dv && L.dvs % 4 == 0, "dvs %d dv %d cs %d", L.dvs, dv, cs);
        CHECK(L.P >= 1 && L.P <= 32 && (L.P & (L.P - 1)) == 0, "P %d", L.P);
        CHECK(L.P * L.dvs <= 256, "P %d dvs %d", L.P, L.dvs);
        CHECK(L.P == 32 || 2 * L.P * L.dvs > 256, "P %d not maximal for dvs %d", L.P, L.dvs);
        CHECK(L.ldT >= L.dvs && L.ldT - L.dvs < 32 && L.ldT % 4 == 0, "ldT %d dvs %d", L.ldT, L.dvs);
        const size_t up4Rm = (size_t)(R * m + 3) / 4 * 4;
        const size_t off[] = {L.skt, L.sqt, L.smu, L.sT, L.ssk, L.ssv, L.sKe, L.sVe, L.sQ, L.sL, L.sF,
                              L.sU, L.sRho, L.sE, L.sMr, L.sZh, L.sZl, L.sS, L.sRow, L.total};
        const size_t len[] = {(size_t)m * d, (size_t)m * d, (size_t)(m * m + 3) / 4 * 4, (size_t)m * L.ldT,
                              (size_t)ns * d, (size_t)ns * L.dvs, (size_t)R * d, (size_t)R * L.dvs, (size_t)R * d,
                              up4Rm, up4Rm, up4Rm, up4Rm, up4Rm, up4Rm, up4Rm, up4Rm,
                              (size_t)(R * ns + 3) / 4 * 4, (size_t)4 * R};
        CHECK(off[0] == 0, "first part at %zu", off[0]);
        for (int i = 0; i < 19; ++i) {
            CHECK(off[i] % 4 == 0, "part %d at float %zu", i, off[i]);
            CHECK(off[i + 1] == off[i] + len[i], "part %d: %zu + %zu != %zu", i, off[i], len[i], off[i + 1]);
        }
        CHECK(short_smem_floats(a) == L.total, "total");
        if (L.total * 4 > max_bytes && L.total * 4 <= 227 * 1024) max_bytes = L.total * 4;
        // value-sum step: thread tid = t * P + pi owns column t (t < dvs) and
        // landmarks pi, pi + P, ...; its reads of T[b][t] within a warp
        for (int w = 0; w < 8; ++w) {
            std::map<int, std::set<long>> bank;
            for (int l = 0; l < 32; ++l) {
                const int tid = 32 * w + l, t = tid / L.P, pi = tid % L.P;
                if (t >= L.dvs || pi >= m) continue;
                const long addr = (long)pi * L.ldT + t;
                bank[(int)(addr % 32)].insert(addr);
            }
            size_t degree = 0;
            for (auto &kv : bank) degree = kv.second.size() > degree ? kv.second.size() : degree;
            if (L.P <= 8) CHECK(degree <= 1, "P %d dvs %d ldT %d: %zu-way bank conflict", L.P, L.dvs, L.ldT, degree);
            else CHECK(degree <= 4, "P %d dvs %d: %zu-way", L.P, L.dvs, degree);
        }
        // every column has its threads
        CHECK(256 / L.P >= L.dvs, "columns %d threads %d", L.dvs, 256 / L.P);
    }
    printf("cases %ld largest fitting layout %zu bytes failures %d\n", cases, max_bytes, failures);
    return failures ? 1 : 0;
}
"""


def test_short_far_kernel_layout(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    src = tmp_path / "short_layout.cu"
    src.write_text(DRIVER)
    exe = tmp_path / "short_layout"
    csrc = os.path.join(ROOT, "sliding_window_landmark_gb300", "csrc")
    subprocess.run([nvcc, "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a", "-I", csrc,
                    "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True, capture_output=True, timeout=300)
    run = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0, run.stdout + run.stderr
    assert "failures 0" in run.stdout, run.stdout
