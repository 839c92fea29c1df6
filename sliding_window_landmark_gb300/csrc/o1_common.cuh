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
#define O1_FB_PLANES 5
#define O1_MAX_D 256
#define O1_MAX_DV 256
#define O1_MAX_M 64
#define O1_MAX_HPG 16
#define O1_MAX_NS 64
#define O1_MAX_W (1 << 20)
#define O1_TC_BN 128           // keys per tile of the tensor-core window path
#define O1_TC_MIN_WINDOW 512   // narrower windows take the fp32 window kernel

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
// keys; per head: landmark queries, mu and the far field (M, Z, T).
struct O1Layout {
    size_t hdr, meta, ring_k, ring_v, sink_k, sink_v, kt, qt, mu, M, Z, T, total;
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
    L.T = off;      off += o1_al256(nh * m * dv * 4);
    L.total = off;
    return L;
}

// A chunk call's scratch for up to `cap` rows per pass (nsub = reference
// blocks of O1_SUB rows):
//   qr [cap][nh][d]  rotated queries        kr [cap][G][d]  rotated keys
//   E  [nh][m][cap]  per row, exp(l - block max) of the key it evicts
//   P  [nh][m][cap]  per row, the in-block prefix of E
//   Fb [O1_FB_PLANES][nh][m][nsub] per block: local max, local mass (from
//                    the block kernel), running max M_c, R_c Z_{c-1} and
//                    the factor exp(local max - M_c) (from the scan); then
//                    [2][nh][m] the far (M, Z) entering the pass
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
struct O1Scratch {
    size_t qr, kr, E, P, Fb, Tp, fh, sh, sn, Xk, XvT, Qs, Sp, total;
    int cap, nsub, nxp;
};

// The tensor-core window path: d in 64-wide chunks (one 128-byte swizzle row
// of fp16), at most 256 (Q_hi and Q_lo take 2 x 64 KB of shared memory at
// d = 256 and leave three 32 KB ring slots), dv a multiple of 32 (TMEM load
// width) up to 256 (O fills TMEM columns 0..255, the two S buffers
// 256..511), and a window wide enough to pay for the panel gather.
static inline bool o1_tc_supported(const o1_geom &g) {
    return g.d % 64 == 0 && g.d <= 256 && g.dv % 32 == 0 && g.dv <= 256 && g.window >= O1_TC_MIN_WINDOW;
}

// Keys per group in the fp16 panels: the ring, the pass's rows, one tile of
// slack for the last tile's overhang, rounded to 8 (16-byte rows of XvT).
static inline int o1_tc_nxp(const o1_geom &g, int cap) { return (g.window + cap + O1_TC_BN + 7) & ~7; }

static inline O1Scratch o1_scratch_layout(const o1_geom &g, int cap) {
    const size_t G = g.groups, nh = (size_t)g.groups * g.heads_per_group, d = g.d, dv = g.dv,
                 m = g.landmarks;
    O1Scratch S;
    S.cap = cap;
    S.nsub = (cap + O1_SUB - 1) / O1_SUB;
    size_t c = (size_t)cap, ns = (size_t)S.nsub, off = 0;
    S.qr = off; off += o1_al256(c * nh * d * 4);
    S.kr = off; off += o1_al256(c * G * d * 4);
    S.E = off;  off += o1_al256(nh * m * c * 4);
    S.P = off;  off += o1_al256(nh * m * c * 4);
    S.Fb = off; off += o1_al256((O1_FB_PLANES * ns + 2) * nh * m * 4);
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
    S.total = off;
    return S;
}

// Far blocks of the one-row path per head, each over dv / O1_TOK_FS value
// columns (rounded up to a multiple of 4). More than one block per head
// measured slower: each recomputes the landmark part, and the shares of T are
// strided rows that a bulk copy cannot bring in whole.
#define O1_TOK_FS 1
__host__ __device__ inline int o1_tok_far_cols(int dv) { return (dv + 4 * O1_TOK_FS - 1) / (4 * O1_TOK_FS) * 4; }
// The far record per head: (c_f, D, have, evicted, numerator [dv], M' [m], Z' [m]).
static inline size_t o1_tok_far_stride(const o1_geom &g) { return 4 + (size_t)g.dv + 2 * (size_t)g.landmarks; }

// Scratch of the one-row path: near partials per (group, key slice, head),
// the value sums [dv] in `part` and (max, sum) in `pml`; the far record per
// head; the row's rotated key per group.
// KC keys per slice (a multiple of 8), NC slices per group, sized for the
// longest near set (sinks + window) so that all groups' slices make about
// 136 blocks (one wave with the far blocks), and capped so that a slice fits
// in shared memory.
struct O1TokScratch {
    size_t part, pml, farp, kcur, total;
    int KC, NC;
};

static inline O1TokScratch o1_tok_layout(const o1_geom &g) {
    const size_t G = g.groups, nh = (size_t)g.groups * g.heads_per_group, dv = g.dv, d = g.d;
    const long long nmax = (long long)g.sinks + g.window;
    long long kc = (nmax * (long long)G + 135) / 136;
    kc = kc < 8 ? 8 : (kc + 7) / 8 * 8;
    // a slice's keys, values, scores and partial dots (8 per key and head)
    // stay within 227 KB of shared memory, rows padded by 4 floats
    const long long kmax = ((227 * 1024 / 4) - (long long)(g.heads_per_group + 1) * (g.d + 4) - 2 * g.heads_per_group) /
                           ((long long)g.d + 4 + g.dv + 9 * g.heads_per_group) / 8 * 8;
    if (kc > kmax) kc = kmax;
    O1TokScratch S;
    S.KC = (int)kc;
    S.NC = (int)((nmax + kc - 1) / kc);
    size_t off = 0;
    S.part = off; off += o1_al256(G * S.NC * g.heads_per_group * dv * 4);
    S.pml = off;  off += o1_al256(G * S.NC * g.heads_per_group * 2 * 4);
    S.farp = off; off += o1_al256(nh * o1_tok_far_stride(g) * 4);
    S.kcur = off; off += o1_al256(G * d * 4);
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
    float *M, *Z, *T;
    // this pass's rows
    const float *q, *k, *v, *gate;
    float *out;
    int R, nsub;
    int commit;   // 0: attend only, the state is left as it was (speculative verify)
    int exact;    // 1: sinks + window only, no far field (the exact-attention comparator)
    // scratch
    float *qr, *kr, *E, *P, *Fb, *Tp, *fh, *sh, *sn;
    int cap;
    // tensor-core window path (tc = 1): fp16 panels of nxp keys per group
    unsigned short *Xk, *XvT, *Qs;
    int nxp, tc;
    float *Sp;   // short-pass window partials (null when the layout has none)
    // one-row path scratch
    float *part, *pml, *farp, *kcur;
    int KC, NC;
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

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

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

// Launchers (o1_chunk.cu). Each returns cudaPeekAtLastError() after its launches.
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
