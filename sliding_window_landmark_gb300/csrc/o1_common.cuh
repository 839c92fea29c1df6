// Internals shared by the library's translation units: the device layout of a
// state and of a call's scratch, the kernel argument block, and block-level
// helpers. Nothing here is part of the C ABI (include/o1.h is).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "o1.h"

#define O1_MAGIC 0x4C53314Fu   // "O1SL"
#define O1_VERSION 1u
#define O1_SUB 64              // rows of one far-field reference block
// Short passes (R >= 2, R * hpg <= O1_SMALL_NQ query vectors): the window
// split over at most O1_SMALL_NS key slices per group
#define O1_SMALL_NQ 64
#define O1_SMALL_NS 64
// planes of the per-block far statistics (scratch Fb)
#define O1_FB_LMAX 0
#define O1_FB_LSUM 1
#define O1_FB_MC 2
#define O1_FB_BASE 3
#define O1_FB_FAC 4
#define O1_FB_BASELO 5
#define O1_FB_PLANES 6
#define O1_MAX_D 256
#define O1_MAX_DV 256
#define O1_MAX_M 64
#define O1_MAX_HPG 16
#define O1_MAX_NS 64
#define O1_MAX_W (1 << 20)
#define O1_TC_BN 128           // keys per tile of the tensor-core window path
#define O1_TC_BM 128           // query rows per CTA of the tensor-core window path
#define O1_SHORT_ROWS 16       // passes up to this many rows take the short far kernel
#define O1_TC_MIN_WINDOW 512   // narrower windows take the fp32 window kernel
// Clock cycles an in-kernel wait may spin before the kernel gives up (about
// 2 s at the maximum SM clock). Drains of copies or MMAs already in flight
// always use this limit; the first waits of a call use O1Args::wait_cycles.
#define O1_WAIT_CYCLES_FULL 4000000000LL

// First bytes of a state buffer.
struct O1Header {
    uint32_t magic;
    uint32_t version;
    o1_geom geom;
    int64_t pos;                       // absolute position of the next row
    uint32_t ticket;                   // arrival counter of last-block commits; 0 between calls
    uint32_t flags;
    float inv_freq[O1_MAX_D / 2];      // rotary inverse frequencies (f32)
};

static inline size_t o1_al256(size_t x) { return (x + 255) & ~(size_t)255; }

// Byte offsets of a state's parts. Per group: meta, ring, sinks, landmark
// keys; per head: landmark queries, mu and the far field (M, Z, T). The far
// mass Z is a sum over every evicted key and grows for as long as the layer
// runs, so it is kept as an unevaluated pair Z + Zlo (Zlo the rounding error
// of Z, |Zlo| <= ulp(Z) / 2) and its recurrence is taken in float-float: an f32
// running sum drifts by about one rounding per update, and signed landmark
// coefficients can cancel the far mass D = sum_b gain_b Z_b down to a small
// fraction of its terms, which magnifies that drift in the output.
// Last come the one-row path's arrival counters (one per head, then one for
// the whole step; G more are kept free), zero between calls.
struct O1Layout {
    size_t hdr, meta, ring_k, ring_v, sink_k, sink_v, kt, qt, mu, M, Z, Zlo, T, tick, total;
};

static inline O1Layout o1_layout(const o1_geom &g) {
    const size_t G = g.groups, nh = (size_t)g.groups * g.heads_per_group, d = g.d, dv = g.dv,
                 ns = g.sinks, w = g.window, m = g.landmarks;
    O1Layout L;
    size_t off = 0;
    L.hdr = off;    off += o1_al256(sizeof(O1Header));
    L.meta = off;   off += o1_al256(G * 4 * sizeof(uint32_t));
    L.ring_k = off; off += o1_al256(G * w * d * 4);
    L.ring_v = off; off += o1_al256(G * w * dv * 4);
    L.sink_k = off; off += o1_al256(G * ns * d * 4);
    L.sink_v = off; off += o1_al256(G * ns * dv * 4);
    L.kt = off;     off += o1_al256(G * m * d * 4);
    L.qt = off;     off += o1_al256(nh * m * d * 4);
    L.mu = off;     off += o1_al256(nh * m * m * 4);
    L.M = off;      off += o1_al256(nh * m * 4);
    L.Z = off;      off += o1_al256(nh * m * 4);
    L.Zlo = off;    off += o1_al256(nh * m * 4);
    L.T = off;      off += o1_al256(nh * m * dv * 4);
    L.tick = off;   off += o1_al256((nh + G + 1) * 4);
    L.total = off;
    return L;
}

// A chunk call's scratch for up to `cap` rows per pass (nsub = reference
// blocks of O1_SUB rows):
//   qr [cap][nh][d]  rotated queries        kr [cap][G][d]  rotated keys
//   E  [nh][m][ldc]  per row, exp(l - block max) of the key it evicts
//   P  [nh][m][ldc]  per row, the in-block prefix of E
//                    (ldc = cap rounded up to 4: rows of 16-byte multiples)
//   Fb [O1_FB_PLANES][nh][m][nsub] per block: local max, local mass (from
//                    the block kernel), running max M_c, R_c Z_{c-1} and
//                    the factor exp(local max - M_c) (from the scan), and
//                    the low part of R_c Z_{c-1}; then [3][nh][m] the far
//                    (M, Z, Zlo) entering the pass
//   Tp [nsub][nh][m][dv]  far value sums: increments relative to the block
//                         max, then the value sum entering each block,
//                         rescaled to its running max
//   fh [cap][nh] x 4      per row-head window header, written by the window
//                         kernel: (reference c_w, mass l, true max, -), the
//                         window numerator being in `out` relative to c_w
//   sh [cap][nh] x 4      per row-head side header (c_s, side mass, -, -)
//   sn [cap][nh][dv]      side numerator (sinks + far field), relative to c_s
// and, when the tensor-core window path serves the geometry, the window key
// sequence as fp16 hi / lo panels (nxp keys per group, zero past the end)
// and the rotated queries as fp16 hi / lo:
//   Xk  [2][G][nxp][d]    XvT [2][G][dv][nxp]    Qs [2][cap][nh][d]
// and, for passes of 2 .. O1_SMALL_NQ / hpg rows, the window partials
//   Sp  [G][O1_SMALL_NS][O1_SMALL_NQ][dv] value sums, then [..][2] (max, sum)
// and, for tensor-core passes split over key ranges (o1_wsplit), the window
// numerators and headers of splits 1 .. S-1 (split 0 writes `out` and fh):
//   Wp  [S-1][R][nh][dv], then [S-1][R][nh][4]
struct O1Scratch {
    size_t qr, kr, E, P, Fb, Tp, fh, sh, sn, Xk, XvT, Qs, Sp, Wp, total;
    int cap, ldc, nsub, nxp;
};

// The tensor-core window path: d in 64-wide chunks (one 128-byte swizzle row
// of fp16), at most 256 (Q_hi and Q_lo take 2 x 64 KB of shared memory at
// d = 256 and leave three 32 KB ring slots), dv a multiple of 32 (TMEM load
// width) up to 256 (O fills TMEM columns 0..255, the two S buffers
// 256..511), and a window wide enough to pay for the panel gather.
static inline bool o1_tc_supported(const o1_geom &g) {
    return g.d % 64 == 0 && g.d <= 256 && g.dv % 32 == 0 && g.dv <= 256 && g.window >= O1_TC_MIN_WINDOW;
}

// Key splits of the tensor-core window kernel for a pass of R rows. A pass
// with fewer CTAs (row blocks x heads) than the GPU has SMs splits each row
// block's key tiles over up to S CTAs, so that short passes (a 64-row chunk
// holds one row block a head) still fill the GPU; the splits' partials meet
// in the merge under one exponent. S stays within the key tiles a row block
// can have.
static inline int o1_wsplit(const o1_geom &g, int R) {
    if (!o1_tc_supported(g) || R < 2) return 1;
    const int ctas = ((R + O1_TC_BM - 1) / O1_TC_BM) * g.groups * g.heads_per_group;
    if (ctas >= 148) return 1;
    const int tmax = (g.window + O1_TC_BM + O1_TC_BN - 1) / O1_TC_BN + 1;
    const int S = (148 + ctas - 1) / ctas;
    return S < tmax ? S : tmax;
}

// Keys per group in the fp16 panels: the ring, the pass's rows, one tile of
// slack for the last tile's overhang, rounded to 8 (16-byte rows of XvT).
static inline int o1_tc_nxp(const o1_geom &g, int cap) { return (g.window + cap + O1_TC_BN + 7) & ~7; }

static inline O1Scratch o1_scratch_layout(const o1_geom &g, int cap) {
    const size_t G = g.groups, nh = (size_t)g.groups * g.heads_per_group, d = g.d, dv = g.dv,
                 m = g.landmarks;
    O1Scratch S;
    S.cap = cap;
    S.ldc = (cap + 3) & ~3;
    S.nsub = (cap + O1_SUB - 1) / O1_SUB;
    size_t c = (size_t)cap, ns = (size_t)S.nsub, off = 0;
    S.qr = off; off += o1_al256(c * nh * d * 4);
    S.kr = off; off += o1_al256(c * G * d * 4);
    S.E = off;  off += o1_al256(nh * m * (size_t)S.ldc * 4);
    S.P = off;  off += o1_al256(nh * m * (size_t)S.ldc * 4);
    S.Fb = off; off += o1_al256((O1_FB_PLANES * ns + 3) * nh * m * 4);
    S.Tp = off; off += o1_al256(ns * nh * m * dv * 4);
    S.fh = off; off += o1_al256(c * nh * 4 * 4);
    S.sh = off; off += o1_al256(c * nh * 4 * 4);
    S.sn = off; off += o1_al256(c * nh * dv * 4);
    S.nxp = o1_tc_supported(g) ? o1_tc_nxp(g, cap) : 0;
    const size_t nx = (size_t)S.nxp;
    S.Xk = off;  off += o1_al256(2 * G * nx * d * 2);
    S.XvT = off; off += o1_al256(2 * G * dv * nx * 2);
    S.Qs = off;  off += o1_al256(S.nxp ? 2 * c * nh * d * 2 : 0);
    // short passes: window partials per (group, key slice, query vector),
    // present from two rows up (a one-row pass never takes that path)
    S.Sp = off;  off += o1_al256(cap >= 2 ? G * O1_SMALL_NS * O1_SMALL_NQ * (dv + 2) * 4 : 0);
    // split partials: the most (S - 1) x R over the passes this scratch can
    // run (S falls as the row blocks grow)
    size_t wrows = 0;
    for (int nrb = 1; (size_t)(nrb - 1) * O1_TC_BM < c; ++nrb) {
        const int R = (int)(c < (size_t)nrb * O1_TC_BM ? c : (size_t)nrb * O1_TC_BM);
        const int Sw = o1_wsplit(g, R);
        if (Sw <= 1) break;
        const size_t wr = (size_t)(Sw - 1) * R;
        wrows = wr > wrows ? wr : wrows;
    }
    S.Wp = off;  off += o1_al256(wrows * nh * (dv + 4) * 4);
    S.total = off;
    return S;
}

// The one-row path runs as one launch of about one wave of CTAs
// (O1_TOK_CTAS): far chunks, one per (head, MB landmarks), NF per head, and
// near slices, one per (group, KC keys of the near set), NC per group, sized
// so that their bytes are about even. Each CTA's shared memory stays under
// O1_TOK_SMEM_CAP, so that the next step's CTAs fit beside a running step's
// and can start loading under its tail.
#define O1_TOK_CTAS 148
#define O1_TOK_SMEM_CAP (100 * 1024)
#define O1_TOK_MB_MAX 32   // landmarks of a far chunk: one per lane of a warp

// Shared memory (floats) of a near slice and of a far chunk, and of the
// merge scratch that follows either; the kernel carves the same offsets.
// After its own work a CTA may merge heads and commit the step: the merge
// stages what it reads (per head, the NC near value sums of dv floats and
// the NF far records of 4 + dv) in the part of shared memory the work used
// (from the near slice's keys, or the far chunk's landmark queries, up to
// the merge scratch), after the rows' factors [heads][NC + NF]. That part is
// made to hold at least the factors, the far records and one near row per
// head (o1_tok_stage_min). The merge scratch holds 8 scalars per head and
// one slot index per group.
__host__ __device__ inline size_t o1_tok_merge_floats(int hpg, int G) { return (size_t)8 * hpg + G + 4; }
__host__ __device__ inline size_t o1_tok_stage_min(int hpg, int NC, int NF, int dv) {
    return ((size_t)hpg * (NC + NF) + 3) / 4 * 4 + (size_t)hpg * NF * (4 + dv) + (size_t)hpg * dv;
}
// (the key rows onwards also take the 8 warps' value-sum partials, 8 hpg dv)
__host__ __device__ inline size_t o1_tok_near_region(int d, int dv, int hpg, int KC) {
    const size_t r = (size_t)KC * (d + dv) + (size_t)KC * hpg + (size_t)8 * KC * hpg, v = (size_t)8 * hpg * dv;
    return r > v ? r : v;
}
__host__ __device__ inline size_t o1_tok_near_floats(int d, int dv, int hpg, int KC, int NC, int NF, int G) {
    const size_t r = o1_tok_near_region(d, dv, hpg, KC), st = o1_tok_stage_min(hpg, NC, NF, dv);
    return 4 + (size_t)hpg * d + d + dv + (size_t)hpg * dv + (r > st ? r : st) + o1_tok_merge_floats(hpg, G);
}
// (from the landmark queries to the end of the numerator partials; the
// merge scratch after it starts 16-byte aligned, through 3 floats of slack)
__host__ __device__ inline size_t o1_tok_far_region(int d, int dv, int m, int MB) {
    return (size_t)MB * d + (size_t)m * d + (size_t)MB * dv + (size_t)m * MB + 8 * (size_t)m + 8 * (size_t)MB +
           2 * (size_t)m + 8 * (size_t)MB + 256;
}
__host__ __device__ inline size_t o1_tok_far_floats(int d, int dv, int hpg, int m, int MB, int NC, int NF, int G) {
    const size_t r = o1_tok_far_region(d, dv, m, MB), st = o1_tok_stage_min(hpg, NC, NF, dv);
    return 4 + 3 * (size_t)d + 2 * (size_t)dv + (size_t)hpg * dv + (r > st ? r : st) + 3 +
           o1_tok_merge_floats(hpg, G);
}

// Scratch of the one-row path: near partials per (group, head, slice), the
// value sums [dv] in `part` and (max, sum) in `pml` (a head's slices are
// contiguous, for the merge's copies); far records per (head,
// chunk): (c_f of the chunk, -, D high, D low, numerator [dv]); the row's
// rotated key per group, for the commit.
struct O1TokScratch {
    size_t part, pml, farp, kcur, total;
    int KC, NC, NF, MB;
    size_t smem;   // bytes of dynamic shared memory per CTA
};

static inline O1TokScratch o1_tok_layout(const o1_geom &g) {
    const long long G = g.groups, hpg = g.heads_per_group, nh = G * hpg, d = g.d, dv = g.dv, m = g.landmarks;
    const long long nnear = (long long)g.sinks + g.window;
    const double near_bytes = 4.0 * G * nnear * (d + dv);
    const double far_head = 4.0 * m * (d + 2 * dv + m);
    const double beta = (near_bytes + nh * far_head) / O1_TOK_CTAS;
    long long NF = (long long)(far_head / beta + 0.999);
    // every chunk also reads all m landmark keys (m d floats): more chunks
    // than the far bytes over that share only repeat it
    const long long nf_max = (d + 2 * dv + m + d - 1) / d;
    NF = NF > nf_max ? nf_max : NF;
    NF = NF < 1 ? 1 : (NF > m ? m : NF);
    long long MB = (m + NF - 1) / NF;
    if (MB > O1_TOK_MB_MAX) MB = O1_TOK_MB_MAX;
    const long long cap = O1_TOK_SMEM_CAP / 4;
    // the merge's staging depends on NC, which is not known yet: size the
    // far chunk with a bound on it (at most O1_TOK_CTAS slices a group). Chunks
    // stay at 8 landmarks or more: below that the parts every chunk holds
    // whole (landmark keys, gate, merge scratch) dominate, and more chunks
    // only repeat them; such a CTA just takes more than the cap.
    while (MB > 8 && (long long)o1_tok_far_floats((int)d, (int)dv, (int)hpg, (int)m, (int)MB, O1_TOK_CTAS,
                                                   (int)((m + MB - 1) / MB), (int)G) > cap)
        MB = (MB + 1) / 2;
    NF = (m + MB - 1) / MB;
    long long near_ctas = O1_TOK_CTAS - nh * NF;
    if (near_ctas < G) near_ctas = G;
    const long long nc0 = (near_ctas + G - 1) / G;
    long long KC = (nnear + nc0 - 1) / nc0;
    KC = KC < 8 ? 8 : (KC + 7) / 8 * 8;
    if (KC > 256) KC = 256;   // a slice's keys sit in a warp's registers, 8 per lane
    long long NC = (nnear + KC - 1) / KC;
    while (KC > 8 && (long long)o1_tok_near_floats((int)d, (int)dv, (int)hpg, (int)KC, (int)NC, (int)NF, (int)G) > cap) {
        KC -= 8;
        NC = (nnear + KC - 1) / KC;
    }
    O1TokScratch S;
    S.KC = (int)KC;
    S.NC = (int)NC;
    S.NF = (int)NF;
    S.MB = (int)MB;
    const size_t nf = o1_tok_far_floats((int)d, (int)dv, (int)hpg, (int)m, (int)MB, (int)NC, (int)NF, (int)G);
    const size_t nn = o1_tok_near_floats((int)d, (int)dv, (int)hpg, (int)KC, (int)NC, (int)NF, (int)G);
    S.smem = 4 * (nf > nn ? nf : nn);
    size_t off = 0;
    S.part = off; off += o1_al256((size_t)G * NC * hpg * dv * 4);
    S.pml = off;  off += o1_al256((size_t)G * NC * hpg * 2 * 4);
    S.farp = off; off += o1_al256((size_t)nh * NF * (4 + dv) * 4);
    S.kcur = off; off += o1_al256((size_t)G * d * 4);
    S.total = off;
    return S;
}

// Scratch that lets a call run passes of up to `rows` rows, a one-row pass
// (the decode path) included.
static inline size_t o1_scratch_need(const o1_geom &g, int rows) {
    const size_t c = o1_scratch_layout(g, rows).total;
    const size_t t = o1_tok_layout(g).total;
    return c > t ? c : t;
}

// Everything a kernel of one pass needs, by value.
struct O1Args {
    int G, hpg, nh, d, dv, ns, w, m, rect, rotate;
    float scale;
    // state
    O1Header *hdr;
    uint32_t *meta;
    float *ring_k, *ring_v;
    const float *sink_k, *sink_v, *kt, *qt, *mu;
    float *M, *Z, *Zlo, *T;
    uint32_t *tick;   // one-row path: arrival counters [nh + G + 1]
    // this pass's rows
    const float *q, *k, *v, *gate;
    float *out;
    int R, nsub;
    long long wait_cycles;   // limit of the first waits (o1_set_wait_limit); drains use O1_WAIT_CYCLES_FULL
    int commit;   // 0: attend only, the state is left as it was (speculative verify)
    int exact;    // 1: sinks + window only, no far field (the exact-attention comparator)
    int short_no_readout;   // short far pass of a commit: inserts only, no side parts
    int chain_early;        // a short pass: its kernels are chained and scheduled before their predecessor ends
    int commit_rotates;     // a short commit pass without the rotation kernel: the keys are rotated where read
    int far_copy;           // the short far kernel left the new M, Z, Zlo in Fb's entering planes; the ring push stores them
    // scratch
    float *qr, *kr, *E, *P, *Fb, *Tp, *fh, *sh, *sn;
    int cap;   // the row stride of E and P (a multiple of 4)
    // window key splits (o1_wsplit): S, and splits 1 .. S-1's numerators
    // [S-1][R][nh][dv] followed by their headers [S-1][R][nh][4]
    int wsplit;
    float *wpart;
    // tensor-core window path (tc = 1): fp16 panels of nxp keys per group
    unsigned short *Xk, *XvT, *Qs;
    int nxp, tc;
    float *Sp;   // short-pass window partials (null when the layout has none)
    // one-row path scratch and work split
    float *part, *pml, *farp, *kcur;
    int KC, NC, NF, MB;
    size_t tok_smem;
    int tok_prefetch;   // issue the state copies before waiting on the previous kernel
    int tok_commit_only;   // push the row (rotation, far insert, ring, meta) without attending
};

// ---------------------------------------------------------------- helpers

// Rotary cos/sin of pair j at position p: the angle p * inv[j] is formed in
// double (inv is f32), reduced by 2 pi in two parts (Cody-Waite), and its
// sine and cosine are taken in f32 with a first-order correction for the
// reduced angle's rounding.
__device__ __forceinline__ void o1_rope_cs(float inv, long long p, float &c, float &s) {
    const double ang = (double)p * (double)inv;
    const double kq = rint(ang * 0.15915494309189535);   // 1 / (2 pi)
    double red = fma(-kq, 6.283185307179586, ang);        // 2 pi, high part
    red = fma(-kq, 2.4492935982947064e-16, red);          // 2 pi, low part
    const float rf = (float)red;
    const float rl = (float)(red - (double)rf);
    float sf, cf;
    sincosf(rf, &sf, &cf);
    c = cf - sf * rl;
    s = sf + cf * rl;
}

// Float4 chunk c4 of key row `row` (raw, from the caller's k) rotated to
// position p: the rotation k_rope applies, pair (j, j + d/2), done where the
// key is read.
__device__ __forceinline__ float4 o1_rot_chunk(const O1Args &a, const float *row, int c4, long long p) {
    const int half = a.d >> 1;
    float y[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const int j = 4 * c4 + e, lo = j < half ? j : j - half;
        float c = 1.f, s = 0.f;
        if (a.rotate) o1_rope_cs(a.hdr->inv_freq[lo], p, c, s);
        const float x0 = row[lo], x1 = row[lo + half];
        y[e] = j < half ? x0 * c - x1 * s : x1 * c + x0 * s;
    }
    return make_float4(y[0], y[1], y[2], y[3]);
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

// Reduce-scatter over a warp: every lane holds 32 partial values; at the
// step over lane bit b a lane keeps the half of its values that its bit
// selects and adds the partner's copy of that half. After five steps (31
// shuffles) x[0] of lane l is the warp's sum of value l.
__device__ __forceinline__ void warp_reduce_scatter32(float (&x)[32]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int b = 16; b >= 1; b >>= 1) {
        const bool up = lane & b;
#pragma unroll
        for (int i = 0; i < b; ++i) {
            const float send = up ? x[i] : x[i + b];
            const float keep = up ? x[i + b] : x[i];
            x[i] = keep + __shfl_xor_sync(0xffffffffu, send, b);
        }
    }
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// Float-float arithmetic: a value as the unevaluated sum hi + lo of two f32
// (|lo| <= ulp(hi) / 2), about 48 significant bits, from f32 operations only
// (FP64 runs at a small fraction of the f32 rate on this part). The error-free
// transformations are Knuth's TwoSum and the fma-based TwoProduct (Dekker;
// Ogita, Rump and Oishi, "Accurate sum and dot product", 2005); the _rn
// intrinsics keep the compiler from contracting or reordering them.
struct o1_ff {
    float hi, lo;
};
__device__ __forceinline__ o1_ff ff_make(float hi, float lo) {
    o1_ff r;
    r.hi = hi;
    r.lo = lo;
    return r;
}
__device__ __forceinline__ o1_ff ff_two_sum(float a, float b) {
    const float s = __fadd_rn(a, b), bb = __fsub_rn(s, a);
    return ff_make(s, __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb)));
}
__device__ __forceinline__ o1_ff ff_fast_two_sum(float a, float b) {   // |a| >= |b| or a == 0
    const float s = __fadd_rn(a, b);
    return ff_make(s, __fsub_rn(b, __fsub_rn(s, a)));
}
__device__ __forceinline__ o1_ff ff_norm(float hi, float lo) { return ff_two_sum(hi, lo); }
__device__ __forceinline__ o1_ff ff_add(o1_ff a, o1_ff b) {
    const o1_ff s = ff_two_sum(a.hi, b.hi);
    return ff_norm(s.hi, __fadd_rn(s.lo, __fadd_rn(a.lo, b.lo)));
}
__device__ __forceinline__ o1_ff ff_add_f(o1_ff a, float b) {
    const o1_ff s = ff_two_sum(a.hi, b);
    return ff_norm(s.hi, __fadd_rn(s.lo, a.lo));
}
// a * b for a float-float a and an f32 b
__device__ __forceinline__ o1_ff ff_mul_f(o1_ff a, float b) {
    const float p = __fmul_rn(a.hi, b);
    const float e = fmaf(a.hi, b, -p);
    return ff_norm(p, fmaf(a.lo, b, e));
}
// acc + a * b for f32 a and b, the product taken exactly
__device__ __forceinline__ o1_ff ff_fma_f(o1_ff acc, float a, float b) {
    const float p = __fmul_rn(a, b);
    return ff_add(acc, ff_make(p, fmaf(a, b, -p)));
}
__device__ __forceinline__ o1_ff warp_sum(o1_ff x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        x = ff_add(x, ff_make(__shfl_xor_sync(0xffffffffu, x.hi, o), __shfl_xor_sync(0xffffffffu, x.lo, o)));
    return x;
}
__device__ __forceinline__ bool ff_nonneg(o1_ff x) { return x.hi > 0.f || (x.hi == 0.f && x.lo >= 0.f); }

// The ring window of group g at the start of a pass: len0 keys in logical
// order from slot head0; wg = the group's window (meta slot 3).
struct O1Meta {
    int len0, head0, farl0, wg;
};

__device__ __forceinline__ O1Meta o1_meta(const O1Args &a, int g) {
    O1Meta mt;
    mt.len0 = (int)a.meta[g * 4 + 0];
    mt.head0 = (int)a.meta[g * 4 + 1];
    mt.farl0 = (int)a.meta[g * 4 + 2];
    mt.wg = (int)a.meta[g * 4 + 3];
    return mt;
}

// Key x of the sequence X = [ring in logical order] ++ [this pass's rows]:
// the rotated key and the value.
__device__ __forceinline__ const float *o1_key(const O1Args &a, int g, int x, const O1Meta &mt) {
    return x < mt.len0 ? a.ring_k + ((size_t)g * a.w + (mt.head0 + x) % mt.wg) * a.d
                       : a.kr + ((size_t)(x - mt.len0) * a.G + g) * a.d;
}

__device__ __forceinline__ const float *o1_val(const O1Args &a, int g, int x, const O1Meta &mt) {
    return x < mt.len0 ? a.ring_v + ((size_t)g * a.w + (mt.head0 + x) % mt.wg) * a.dv
                       : a.v + ((size_t)(x - mt.len0) * a.G + g) * a.dv;
}

// Block-level fp32 products on shared-memory tiles, 256 threads, a 64 x 64
// output held as 4 x 4 per thread (rows ty + 16 i, columns tx + 16 j).
//   nt: c[i][j] += sum_k A[row_i][k] * B[col_j][k]   (both K-contiguous)
//   nn: c[i][j] += sum_k A[row_i][k] * B[k][col_j]
// Odd leading dimensions keep the column reads free of bank conflicts.
__device__ __forceinline__ void blk_nt(float (&c)[4][4], const float *A, int lda, const float *B,
                                       int ldb, int K) {
    const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
#pragma unroll 4
    for (int k = 0; k < K; ++k) {
        float av[4], bv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) av[i] = A[(ty + 16 * i) * lda + k];
#pragma unroll
        for (int j = 0; j < 4; ++j) bv[j] = B[(tx + 16 * j) * ldb + k];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) c[i][j] = fmaf(av[i], bv[j], c[i][j]);
    }
}

__device__ __forceinline__ void blk_nn(float (&c)[4][4], const float *A, int lda, const float *B,
                                       int ldb, int K) {
    const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
#pragma unroll 4
    for (int k = 0; k < K; ++k) {
        float av[4], bv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) av[i] = A[(ty + 16 * i) * lda + k];
#pragma unroll
        for (int j = 0; j < 4; ++j) bv[j] = B[k * ldb + tx + 16 * j];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) c[i][j] = fmaf(av[i], bv[j], c[i][j]);
    }
}

__device__ __forceinline__ void blk_zero(float (&c)[4][4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) c[i][j] = 0.f;
}

// Per-device once: a kernel's dynamic shared memory limit is a setting of the
// current device, so each launcher keeps one bit per device (up to 64) in
// `mask`, set after its attributes are. Two host threads racing on a
// device's first call both set them (the setting is idempotent); none
// launches before they are set.
static inline bool o1_attrs_needed(const unsigned long long *mask, unsigned long long *bit) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        *bit = 0;
        return true;
    }
    *bit = 1ull << dev;
    return !(__atomic_load_n(mask, __ATOMIC_ACQUIRE) & *bit);
}
static inline void o1_attrs_done(unsigned long long *mask, unsigned long long bit) {
    __atomic_fetch_or(mask, bit, __ATOMIC_RELEASE);
}

// Chained launches (programmatic dependent launch), used in short passes
// (at most O1_SHORT_ROWS rows: the key-slice window kernels, the short
// commit pass; O1Args::chain_early). A kernel launched by o1_launch_chained
// with `chained` set may be scheduled while the previous kernel of its
// stream is still running, so every kernel that can be launched that way
// calls o1_chain_wait() before it touches global memory; the wait returns
// once that kernel has completed and its writes are visible (and at once
// after a plain launch). Since every chained kernel waits, a chain completes
// in order. The first kernel of a pass on a stream, and every kernel behind
// an event wait, is launched plainly. o1_chain_release() lets the next
// chained kernel be scheduled before this one ends; the kernels that can
// end a pass never call it, because a one-row step launched after them reads
// the state ahead of its own wait. Longer passes launch plainly: chaining
// them measured slower (a 24-layer stack of 64-row chunks 40.7 -> 48.9 ms,
// a 4096-row prompt with early release 0.370 -> 0.396 ms).
__device__ __forceinline__ void o1_chain_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void o1_chain_release() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... P, typename... A>
static inline void o1_launch_chained(bool chained, void (*k)(P...), dim3 grid, dim3 block, size_t smem,
                                     cudaStream_t st, A... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = chained ? 1 : 0;
    cudaLaunchKernelEx(&cfg, k, args...);
}

// The short far kernel (k_side_short, o1_chunk.cu): CTAs per head (the value
// columns split over up to 4) and its shared-memory layout.
__host__ __device__ inline int short_col_splits(const O1Args &a) {
    for (int cs = 4; cs > 1; cs >>= 1)
        if (a.nh * cs <= 148 && a.dv % (4 * cs) == 0) return cs;
    return 1;
}

// Shared memory of k_side_short, in floats; every part starts on 16 bytes.
struct ShortLayout {
    int dvs;   // value columns of this CTA
    int P;     // threads per value column in step 4 (a power of two, at most 32)
    int ldT;   // row stride of T: P lanes on P landmarks of one column hit P different banks
    size_t skt, sqt, smu, sT, ssk, ssv, sKe, sVe, sQ, sL, sF, sU, sRho, sE, sMr, sZh, sZl, sS, sRow, total;
};
__host__ __device__ inline size_t short_up4(size_t x) { return (x + 3) / 4 * 4; }
__host__ __device__ inline ShortLayout short_layout(const O1Args &a) {
    ShortLayout L;
    L.dvs = a.dv / short_col_splits(a);
    L.P = 1;
    while (L.P < 32 && 2 * L.P * L.dvs <= 256) L.P *= 2;
    const int off = L.P >= 8 ? 4 : 32 / L.P;   // stride = off (mod 32), a multiple of 4
    L.ldT = L.dvs + ((off - L.dvs) % 32 + 32) % 32;
    const size_t m = a.m, d = a.d, dvs = L.dvs, ns = a.ns, R = a.R;
    size_t o = 0;
    L.skt = o;  o += m * d;                // [m][d]   landmark keys of the group
    L.sqt = o;  o += m * d;                // [m][d]   landmark queries of the head
    L.smu = o;  o += short_up4(m * m);     // [m][m]
    L.sT = o;   o += m * L.ldT;            // [m][ldT] far value sums (this slice)
    L.ssk = o;  o += ns * d;               // [ns][d]
    L.ssv = o;  o += ns * dvs;             // [ns][dvs]
    L.sKe = o;  o += R * d;                // [R][d]   the key each row evicts
    L.sVe = o;  o += R * dvs;              // [R][dvs] and its value
    L.sQ = o;   o += R * d;                // [R][d]   the rows' rotated queries
    L.sL = o;   o += short_up4(R * m);     // [R][m]   insert logits
    L.sF = o;   o += short_up4(R * m);     // [R][m]   far scores, then e^{f - F}
    L.sU = o;   o += short_up4(R * m);     // [R][m]   u, then the gains
    L.sRho = o; o += short_up4(R * m);     // [R][m]   the inserts' rescales
    L.sE = o;   o += short_up4(R * m);     //          and weights
    L.sMr = o;  o += short_up4(R * m);     // [R][m]   M after each row's insert
    L.sZh = o;  o += short_up4(R * m);     //          and Z, high
    L.sZl = o;  o += short_up4(R * m);     //          and low part
    L.sS = o;   o += short_up4(R * ns);    // [R][ns]  sink scores, then weights
    L.sRow = o; o += 4 * R;                // [R][4]   F, e^{c_f - c_s} (0: no far part)
    L.total = o;
    return L;
}
__host__ __device__ inline size_t short_smem_floats(const O1Args &a) { return short_layout(a).total; }

// Launchers (o1_chunk.cu). Each returns cudaGetLastError() after its launches.
// `ev` may be null; otherwise 2 * O1_NUM_STAGES events, one before and one after each stage.
cudaError_t o1_launch_pass(const O1Args &a, cudaStream_t st, cudaEvent_t const *ev = nullptr);
cudaError_t o1_launch_init(const O1Args &a, cudaStream_t st);
// Rewind `rows` ring pushes of every group (meta and position).
cudaError_t o1_launch_back(const O1Args &a, int rows, cudaStream_t st);
// The state-advancing stages alone over a.R rows whose keys and values are
// in a.k and a.v (a.q unused): rotation of the keys, far insert, ring push,
// meta and position.
cudaError_t o1_launch_commit_pass(const O1Args &a, cudaStream_t st);
// Tensor-core window path (o1_near_tc.cu): panel gather, then the window
// attention with the side merge and the gate.
cudaError_t o1_launch_gather_tc(const O1Args &a, cudaStream_t st);
cudaError_t o1_launch_near_tc(const O1Args &a, cudaStream_t st);
// One row (o1_token.cu): main kernel + merge kernel.
cudaError_t o1_launch_token(const O1Args &a, cudaStream_t st);
