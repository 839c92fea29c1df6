// The chunk path of a sealed O(1) layer: one pass over R rows.
//
// The method is the one of "cortiq-engine 0.8.51 src/gpu_wgpu/o1_batch.rs":
// per row, sinks + the row's ring window + the landmark far field; the state
// moves by rope, far insert, ring push (module doc). The pages run it as five
// dispatches per 64-row sub-chunk (o1b_far_e, o1b_attend, o1b_far_commit,
// o1b_ring_commit, o1b_meta), each sub-chunk waiting for the last. Here the
// whole pass is parallel, because only the far field is sequential and its
// per-block partials compose associatively:
//
//  1. k_rope         rotate q and k of every row (dory.rs, dory_prep)
//  2. k_far_logits   l = scale qt_b . k_e for every key the pass evicts
//                    (o1b_far_e's dot, all blocks at once)
//  3. k_far_scan     per (head, landmark): block max M_c, rescale R_c,
//                    E = exp(l - M_c), far-mass prefix P per row (o1b_far_e's
//                    max / rescale / prefix, as a scan over the blocks)
//  4. k_far_dT       per block: sum_j E_bj v_ev(j)  (o1b_far_commit's sum)
//  5. k_far_tscan    T entering each block, rescaled to its max
//                    (o1b_far_commit's recurrence T <- R T + dT, as a scan)
//  6. k_side_readout per row: the sinks and the far field (landmark scores,
//                    u = e^{f-F} mu, gains, far mass and numerator) under one
//                    exponent (o1b_attend's sink and far parts)
//  7. k_gather_tc    (tensor-core geometries) the window key sequence as
//                    fp16 hi / lo panels (o1_near_tc.cu)
//  8. k_near_tc      the sliding window on the tensor cores (o1b_attend's
//     or k_near      window part); k_near is the fp32 version for the other
//                    geometries
//  9. k_merge        window and side parts under one exponent, the 1e-30
//                    floor, the gate (o1b_attend's normalisation; dory_gate1)
// 10. k_commit       ring rows and meta (o1b_ring_commit, o1b_meta)
// Stages 2-6 and 7-8 share no data; they run on two streams.
//
// Keys are indexed in X = [ring, oldest first] ++ [this pass's rows]: row r
// sees X[max(0, len0 + r + 1 - wg) .. len0 + r] and evicts X[r - j0] once
// r >= j0 = wg - len0 (o1b_far_e: "ring logical index j - j0"). That indexing
// also covers a pass whose rows evict keys pushed earlier in the same pass
// (window shorter than a block), which the pages' sub-chunking excludes.
#include <cuda_fp16.h>
#include <math.h>

#include "o1_common.cuh"

// ------------------------------------------------------------------ rope

// One block per row. Thread j < d/2 forms the angle of pair (j, j + d/2)
// once (o1_rope_cs: within a few f32 ulp of the pages' f64-then-f32 table)
// and rotates every query head and every key group with it.
__global__ void k_rope(O1Args a) {
    const int r = blockIdx.x;
    const int half = a.d >> 1;
    const int64_t p = a.hdr->pos + r;
    for (int j = threadIdx.x; j < half; j += blockDim.x) {
        float c = 1.f, s = 0.f;
        if (a.rotate) o1_rope_cs(a.hdr->inv_freq[j], p, c, s);
        // 8 heads' loads ahead of their stores
        for (int h0 = 0; h0 < a.nh; h0 += 8) {
            float x0[8], x1[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const size_t o = ((size_t)r * a.nh + h0 + u) * a.d;
                x0[u] = h0 + u < a.nh ? a.q[o + j] : 0.f;
                x1[u] = h0 + u < a.nh ? a.q[o + j + half] : 0.f;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (h0 + u >= a.nh) break;
                const size_t o = ((size_t)r * a.nh + h0 + u) * a.d;
                const float y0 = x0[u] * c - x1[u] * s, y1 = x1[u] * c + x0[u] * s;
                a.qr[o + j] = y0;
                a.qr[o + j + half] = y1;
                if (a.tc) {
                    // fp16 hi / lo of the rotated query for the tensor-core window path
                    const size_t lo_off = (size_t)a.R * a.nh * a.d;
                    const __half h0v = __float2half_rn(y0), h1v = __float2half_rn(y1);
                    a.Qs[o + j] = __half_as_ushort(h0v);
                    a.Qs[o + j + half] = __half_as_ushort(h1v);
                    a.Qs[lo_off + o + j] = __half_as_ushort(__float2half_rn(y0 - __half2float(h0v)));
                    a.Qs[lo_off + o + j + half] = __half_as_ushort(__float2half_rn(y1 - __half2float(h1v)));
                    if (!(fabsf(y0) < 65504.f && fabsf(y1) < 65504.f)) atomicOr(&a.hdr->flags, (uint32_t)O1_FLAG_FP16_RANGE);
                }
            }
        }
        for (int g = 0; g < a.G; ++g) {
            const size_t o = ((size_t)r * a.G + g) * a.d;
            const float x0 = a.k[o + j], x1 = a.k[o + j + half];
            a.kr[o + j] = x0 * c - x1 * s;
            a.kr[o + j + half] = x1 * c + x0 * s;
        }
    }
}

// ------------------------------------------------------------- far field

// Far logits of the evicted keys: E[gh][b][x] = scale qt[gh][b] . X[x] for
// x < R - j0. Block = (64 evicted keys, head).
__global__ __launch_bounds__(256) void k_far_logits(O1Args a) {
    const int gh = blockIdx.y, g = gh / a.hpg;
    const O1Meta mt = o1_meta(a, g);
    const int j0 = mt.wg - mt.len0;
    const int nev = a.R - j0;
    const int x0 = blockIdx.x * 64;
    if (x0 >= nev) return;
    __shared__ float sA[64 * 33], sB[64 * 33];
    float c[4][4];
    blk_zero(c);
    for (int kc = 0; kc < a.d; kc += 32) {
        for (int idx = threadIdx.x; idx < 64 * 32; idx += 256) {
            const int i = idx >> 5, kk = idx & 31;
            const bool in = kc + kk < a.d;
            sA[i * 33 + kk] = (i < a.m && in) ? a.qt[((size_t)gh * a.m + i) * a.d + kc + kk] : 0.f;
            sB[i * 33 + kk] = (x0 + i < nev && in) ? o1_key(a, g, x0 + i, mt)[kc + kk] : 0.f;
        }
        __syncthreads();
        blk_nt(c, sA, 33, sB, 33, 32);
        __syncthreads();
    }
    const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int b = ty + 16 * i, x = x0 + tx + 16 * j;
            if (b < a.m && x < nev) a.E[((size_t)gh * a.m + b) * a.cap + x] = a.scale * c[i][j];
        }
}

// One warp per (head, landmark query b), sequential over the pass's blocks of
// O1_SUB rows: the far max after each block M_c, the rescale R_c of what came
// before (1 if the max did not move, so an empty field stays empty), E =
// exp(l - M_c) in place of l, and for every row the far mass P = R_c Z +
// (prefix of E within the block).
__global__ __launch_bounds__(256) void k_far_scan(O1Args a) {
    const int wid = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (wid >= a.nh * a.m) return;
    const int gh = wid / a.m, g = gh / a.hpg;
    const O1Meta mt = o1_meta(a, g);
    const int j0 = mt.wg - mt.len0;
    float Mo = a.M[wid], Zo = a.Z[wid];
    float *E = a.E + (size_t)wid * a.cap;
    float *P = a.P + (size_t)wid * a.cap;
    constexpr int NB = 4;   // blocks whose logits are loaded ahead of their stores
    float lq[NB][2];
    for (int c = 0; c < a.nsub; ++c) {
        const int r0 = c * O1_SUB;
        if (c % NB == 0) {
#pragma unroll
            for (int q = 0; q < NB; ++q)
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const int r = (c + q) * O1_SUB + hf * 32 + lane;
                    lq[q][hf] = (r < a.R && r >= j0) ? E[r - j0] : -INFINITY;
                }
        }
        float l[2];
        bool ev[2];
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            const int r = r0 + hf * 32 + lane;
            ev[hf] = r < a.R && r >= j0;
#pragma unroll
            for (int q = 0; q < NB; ++q)
                if (q == c % NB) l[hf] = lq[q][hf];
        }
        const float Mn = fmaxf(Mo, warp_max(fmaxf(l[0], l[1])));
        const float Rf = (Mn == Mo) ? 1.f : expf(Mo - Mn);
        const float base = Rf * Zo;
        float run = 0.f;
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
            const int r = r0 + hf * 32 + lane;
            const float e = ev[hf] ? expf(l[hf] - Mn) : 0.f;
            if (ev[hf]) E[r - j0] = e;
            float incl = e;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float t = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += t;
            }
            if (r < a.R) P[r] = base + (run + incl);
            run += __shfl_sync(0xffffffffu, incl, 31);
        }
        Zo = base + run;
        Mo = Mn;
        if (lane == 0) {
            a.Mc[(size_t)wid * a.nsub + c] = Mn;
            a.Rc[(size_t)wid * a.nsub + c] = Rf;
        }
    }
    if (lane == 0) {
        a.M[wid] = Mo;
        a.Z[wid] = Zo;
    }
}

// Value-sum increment of each block: dT[c][gh][b][t] = sum over the block's
// evicting rows j of E[b][j] v_ev(j)[t]. Block = (block c, head, 64 columns).
__global__ __launch_bounds__(256) void k_far_dT(O1Args a) {
    const int c = blockIdx.x, gh = blockIdx.y, tc = blockIdx.z * 64, g = gh / a.hpg;
    const O1Meta mt = o1_meta(a, g);
    const int j0 = mt.wg - mt.len0;
    const int r0 = c * O1_SUB, nr = min(O1_SUB, a.R - r0);
    float *dst = a.Tp + (size_t)(c * a.nh + gh) * a.m * a.dv;
    const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
    if (max(r0, j0) >= r0 + nr) {   // nothing evicted in this block
        for (int idx = threadIdx.x; idx < a.m * 64; idx += 256) {
            const int b = idx >> 6, t = tc + (idx & 63);
            if (t < a.dv) dst[(size_t)b * a.dv + t] = 0.f;
        }
        return;
    }
    __shared__ float sA[64 * 65], sB[64 * 65];
    for (int idx = threadIdx.x; idx < 64 * 64; idx += 256) {
        const int i = idx >> 6, jj = idx & 63;
        const int r = r0 + jj;
        const bool evj = jj < nr && r >= j0;
        sA[i * 65 + jj] = (i < a.m && evj) ? a.E[((size_t)gh * a.m + i) * a.cap + (r - j0)] : 0.f;
        // row i of B is evicting row r0 + i, column jj is value column tc + jj
        const int ri = r0 + i;
        const bool evi = i < nr && ri >= j0 && tc + jj < a.dv;
        sB[i * 65 + jj] = evi ? o1_val(a, g, ri - j0, mt)[tc + jj] : 0.f;
    }
    __syncthreads();
    float acc[4][4];
    blk_zero(acc);
    blk_nn(acc, sA, 65, sB, 65, 64);
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int b = ty + 16 * i, t = tc + tx + 16 * j;
            if (b < a.m && t < a.dv) dst[(size_t)b * a.dv + t] = acc[i][j];
        }
}

// The value sum entering each block, rescaled to that block's max:
// Tp[c] <- R_c T_{c-1} (what the block's rows read), T_c = R_c T_{c-1} + dT_c;
// the last T is the new state. One thread per (head, landmark, column).
__global__ void k_far_tscan(O1Args a) {
    const size_t n = (size_t)a.nh * a.m * a.dv;
    const size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= n) return;
    const size_t wid = idx / a.dv;
    float T = a.T[idx];
    // 16 blocks' loads issued before their stores (the compiler cannot
    // reorder them itself: the stores may alias later loads for all it knows)
    for (int c0 = 0; c0 < a.nsub; c0 += 16) {
        float rf[16], dT[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int c = c0 + i;
            rf[i] = c < a.nsub ? a.Rc[wid * a.nsub + c] : 1.f;
            dT[i] = c < a.nsub ? a.Tp[(size_t)c * n + idx] : 0.f;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const int c = c0 + i;
            if (c < a.nsub) {
                const float Ts = rf[i] * T;
                a.Tp[(size_t)c * n + idx] = Ts;
                T = Ts + dT[i];
            }
        }
    }
    a.T[idx] = T;
}

// The side part of every row of block c for head gh: the sinks and the far
// field, referenced to one exponent c_s = max(sink scores, c_f) (o1b_attend's
// c_all restricted to these keys; the far half as the pages reference it to
// the block's max):
//   f_a = scale q'.kt_a, F = max f, u_b = sum_a e^{f_a - F} mu[a][b] (rect),
//   c_f = max_b (F + M_c[b]), gain_b = u_b e^{F + M_c[b] - c_f},
//   D = sum_b gain_b P_b(row); the far part is dropped if D < 0 (c_f still
//   enters c_s, as c_all keeps the far max);
//   far numerator = sum_b gain_b (R_c T_{c-1})_b + sum_{evicting j <= row} cf_j v_ev(j),
//   cf_j = sum_b gain_b E_bj;
//   sinks: p_x = e^{scale q'.sink_x - c_s}.
// The side numerator goes to the side buffer sn and (c_s, side mass) to the
// row's side header; c_s = -inf marks a row with no sinks and no far field.
//
// Layout (256 threads, 8 warps). The products are register-tiled with
// float4 shared-memory reads:
//   scores  [64 rows] x [landmarks | sinks] over d, 4 x 4 per thread,
//           k in float4 steps (both operands k-contiguous);
//   side numerator = A6 . B6 in one product of depth K6 = m + 64 + ns:
//           A6 = [gains | in-block coefficients | sink weights] (stored
//           k-major, so a warp's 8 rows are one broadcast float4 pair),
//           B6 = [T entering the block | evicted values | sink values],
//           8 rows x 4 NV columns per thread (warp = 8 rows).
constexpr int SR_LDQ = 36;   // 32-wide k chunk + 4
constexpr int SR_LDA = 68;   // A6 row stride (64 rows + 4)

__host__ __device__ inline void side_layout(const O1Args &a, size_t off[6]) {
    const int nbt = (a.m + a.ns + 63) / 64;
    const int K6 = a.m + 64 + a.ns;
    const size_t r1a = (size_t)64 * SR_LDQ * (1 + nbt), r1b = (size_t)32 * (a.dv + 4);
    off[0] = 0;                                              // A6 [K6][SR_LDA]
    off[1] = off[0] + (size_t)K6 * SR_LDA;                   // R1: score chunks, then B6 chunks
    off[2] = off[1] + (r1a > r1b ? r1a : r1b);               // sS [64][64 nbt + 1]
    off[3] = off[2] + (size_t)64 * (64 * nbt + 1);           // R3: mu, then E [64][65]
    off[4] = off[3] + 64 * 65;                               // F, M_c [64] each
    off[5] = off[4] + 2 * 64;                                // total (floats)
}

__device__ __forceinline__ void fma4x4_k4(float (&c)[4][4], const float4 (&av)[4], const float4 (&bv)[4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            c[i][j] = fmaf(av[i].x, bv[j].x, c[i][j]);
            c[i][j] = fmaf(av[i].y, bv[j].y, c[i][j]);
            c[i][j] = fmaf(av[i].z, bv[j].z, c[i][j]);
            c[i][j] = fmaf(av[i].w, bv[j].w, c[i][j]);
        }
}

template <int NV>
__global__ __launch_bounds__(256, 2) void k_side_readout(O1Args a) {
    extern __shared__ __align__(16) float sm[];
    const int c = blockIdx.x, gh = blockIdx.y, g = gh / a.hpg;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int ty = tid >> 4, tx = tid & 15;
    const O1Meta mt = o1_meta(a, g);
    const int j0 = mt.wg - mt.len0;
    const int r0 = c * O1_SUB, nr = min(O1_SUB, a.R - r0);
    const int m = a.m, d = a.d, dv = a.dv, nh = a.nh, ns = a.ns;
    const bool far_any = mt.farl0 + max(0, r0 + nr - j0) > 0;
    size_t off[6];
    side_layout(a, off);
    const int nbt = (m + ns + 63) / 64;
    const int ldS = 64 * nbt + 1;
    const int K6 = m + 64 + ns;
    float *sA6 = sm + off[0];
    float *sR1 = sm + off[1];
    float *sS = sm + off[2];
    float *sR3 = sm + off[3];
    float *sRow = sm + off[4];
    float *sMc = sRow + 64;

    // 1. scores: columns [0, m) landmarks f_a, [m, m + ns) sinks
    {
        float *sQc = sR1;                    // [64][SR_LDQ]
        float *sBc = sR1 + 64 * SR_LDQ;      // [64 nbt][SR_LDQ]
        float acc[2][4][4];
#pragma unroll
        for (int t = 0; t < 2; ++t) blk_zero(acc[t]);
        const int nrow = 64 * (1 + nbt);
        for (int kc = 0; kc < d; kc += 32) {
            for (int idx = tid; idx < nrow * 8; idx += 256) {
                const int row = idx >> 3, k = kc + 4 * (idx & 7);
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (k < d) {
                    if (row < 64) {
                        if (row < nr) v = *(const float4 *)(a.qr + ((size_t)(r0 + row) * nh + gh) * d + k);
                    } else {
                        const int col = row - 64;
                        if (col < m) {
                            if (far_any) v = *(const float4 *)(a.kt + ((size_t)g * m + col) * d + k);
                        } else if (col < m + ns) {
                            v = *(const float4 *)(a.sink_k + ((size_t)g * ns + col - m) * d + k);
                        }
                    }
                }
                *(float4 *)(sR1 + row * SR_LDQ + 4 * (idx & 7)) = v;
            }
            __syncthreads();
#pragma unroll 2
            for (int k4 = 0; k4 < 8; ++k4) {
                float4 av[4], bv[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) av[i] = *(const float4 *)(sQc + (ty + 16 * i) * SR_LDQ + 4 * k4);
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    if (t < nbt) {
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            bv[j] = *(const float4 *)(sBc + (64 * t + tx + 16 * j) * SR_LDQ + 4 * k4);
                        fma4x4_k4(acc[t], av, bv);
                    }
                }
            }
            __syncthreads();
        }
#pragma unroll
        for (int t = 0; t < 2; ++t)
            if (t < nbt)
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) sS[(ty + 16 * i) * ldS + 64 * t + tx + 16 * j] = a.scale * acc[t][i][j];
    }
    __syncthreads();   // scores complete before any row reads them (step 2 or 4)
    if (far_any) {
        float *sMu = sR3;   // [m][65]
        for (int idx = tid; idx < m * m; idx += 256) {
            const int aa = idx / m, b = idx % m;
            sMu[aa * 65 + b] = a.mu[((size_t)gh * m + aa) * m + b];
        }
        for (int b = tid; b < 64; b += 256) sMc[b] = b < m ? a.Mc[((size_t)gh * m + b) * a.nsub + c] : 0.f;
        __syncthreads();
        // 2. F per row and e^{f - F} (columns [0, m))
        for (int i = warp; i < 64; i += 8) {
            const float v0 = lane < m ? sS[i * ldS + lane] : -INFINITY;
            const float v1 = lane + 32 < m ? sS[i * ldS + lane + 32] : -INFINITY;
            const float F = warp_max(fmaxf(v0, v1));
            if (lane == 0) sRow[i] = F;
            if (lane < m) sS[i * ldS + lane] = expf(v0 - F);
            if (lane + 32 < m) sS[i * ldS + lane + 32] = expf(v1 - F);
        }
        __syncthreads();
        // 3. u = e mu, written back over columns [0, m)
        float acc[4][4];
        blk_zero(acc);
        blk_nn(acc, sS, ldS, sMu, 65, m);
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (tx + 16 * j < m) sS[(ty + 16 * i) * ldS + tx + 16 * j] = acc[i][j];
        __syncthreads();
        // E of this block's evicting rows, referenced to M_c by k_far_scan
        float *sE = sR3;   // [m][65]
        for (int idx = tid; idx < m * 64; idx += 256) {
            const int b = idx >> 6, jj = idx & 63;
            const int r = r0 + jj;
            sE[b * 65 + jj] = (jj < nr && r >= j0) ? a.E[((size_t)gh * m + b) * a.cap + (r - j0)] : 0.f;
        }
    }

    // 4. per row (one warp each): far gains, mass and sign decision, the side
    //    exponent c_s, sink weights, the side mass; gains and sink weights
    //    into A6 (k-major)
    for (int i = warp; i < 64; i += 8) {
        const int r = r0 + i;
        const int farl = mt.farl0 + max(0, r - j0 + 1);
        float g0 = 0.f, g1 = 0.f, cf = -INFINITY, D = 0.f;
        bool have = false;
        if (far_any && i < nr && farl > 0) {
            float u0 = lane < m ? sS[i * ldS + lane] : 0.f;
            float u1 = lane + 32 < m ? sS[i * ldS + lane + 32] : 0.f;
            if (a.rect) {
                u0 = fmaxf(u0, 0.f);
                u1 = fmaxf(u1, 0.f);
            }
            const float F = sRow[i];
            const float cb0 = lane < m ? F + sMc[lane] : -INFINITY;
            const float cb1 = lane + 32 < m ? F + sMc[lane + 32] : -INFINITY;
            cf = warp_max(fmaxf(cb0, cb1));
            g0 = lane < m ? u0 * expf(cb0 - cf) : 0.f;
            g1 = lane + 32 < m ? u1 * expf(cb1 - cf) : 0.f;
            const float p0 = lane < m ? a.P[((size_t)gh * m + lane) * a.cap + r] : 0.f;
            const float p1 = lane + 32 < m ? a.P[((size_t)gh * m + lane + 32) * a.cap + r] : 0.f;
            D = warp_sum(g0 * p0 + g1 * p1);
            have = D >= 0.f;
        }
        const float sx0 = (i < nr && lane < ns) ? sS[i * ldS + m + lane] : -INFINITY;
        const float sx1 = (i < nr && lane + 32 < ns) ? sS[i * ldS + m + lane + 32] : -INFINITY;
        const float smax = warp_max(fmaxf(sx0, sx1));
        const float cs = fmaxf(smax, cf);
        const float w0 = sx0 > -INFINITY ? expf(sx0 - cs) : 0.f;
        const float w1 = sx1 > -INFINITY ? expf(sx1 - cs) : 0.f;
        const float fs = have ? expf(cf - cs) : 0.f;
        const float side = warp_sum(w0 + w1) + fs * D;
        if (lane < m) sA6[lane * SR_LDA + i] = g0 * fs;
        if (lane + 32 < m) sA6[(lane + 32) * SR_LDA + i] = g1 * fs;
        if (lane < ns) sA6[(m + 64 + lane) * SR_LDA + i] = w0;
        if (lane + 32 < ns) sA6[(m + 64 + lane + 32) * SR_LDA + i] = w1;
        if (i < nr && lane == 0)
            *(float4 *)(a.sh + ((size_t)r * nh + gh) * 4) = make_float4(cs, cs > -INFINITY ? side : 0.f, 0.f, 0.f);
    }
    __syncthreads();
    // 5. in-block far coefficients, causal: W[row][jj] = sum_b gain_b(row) E_b(jj)
    //    for jj <= row, into A6 rows m + jj
    if (far_any) {
        const float *sE = sR3;
        float acc[4][4];
        blk_zero(acc);
#pragma unroll 4
        for (int b = 0; b < m; ++b) {
            float av[4], bv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) av[i] = sA6[b * SR_LDA + ty + 16 * i];
#pragma unroll
            for (int j = 0; j < 4; ++j) bv[j] = sE[b * 65 + tx + 16 * j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int row = ty + 16 * i, jj = tx + 16 * j;
                sA6[(m + jj) * SR_LDA + row] = jj <= row ? acc[i][j] : 0.f;
            }
    }
    __syncthreads();

    // 6. side numerator = A6 . B6, B6 rows: T entering the block (b < m), the
    //    evicted values (m + jj), the sink values (m + 64 + x)
    const float *Tp = a.Tp + (size_t)(c * nh + gh) * m * dv;
    const float *sinks_v = a.sink_v + (size_t)g * ns * dv;
    const int kbeg = far_any ? 0 : (ns > 0 ? m + 64 : K6);
    const int ldB = dv + 4, dv4 = dv >> 2;
    float acc6[8][NV][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int v = 0; v < NV; ++v) acc6[i][v][0] = acc6[i][v][1] = acc6[i][v][2] = acc6[i][v][3] = 0.f;
    for (int k0 = kbeg; k0 < K6; k0 += 32) {
        const int kn = min(32, K6 - k0);
        for (int idx = tid; idx < kn * dv4; idx += 256) {
            const int kk = idx / dv4, c4 = idx % dv4, k = k0 + kk;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (k < m) {
                v = *(const float4 *)(Tp + (size_t)k * dv + 4 * c4);
            } else if (k < m + 64) {
                const int jj = k - m, r = r0 + jj;
                if (jj < nr && r >= j0) v = ((const float4 *)o1_val(a, g, r - j0, mt))[c4];
            } else {
                v = *(const float4 *)(sinks_v + (size_t)(k - m - 64) * dv + 4 * c4);
            }
            *(float4 *)(sR1 + kk * ldB + 4 * c4) = v;
        }
        __syncthreads();
#pragma unroll 2
        for (int kk = 0; kk < kn; ++kk) {
            const float4 a0 = *(const float4 *)(sA6 + (k0 + kk) * SR_LDA + 8 * warp);
            const float4 a1 = *(const float4 *)(sA6 + (k0 + kk) * SR_LDA + 8 * warp + 4);
            const float ar[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                const int col = 4 * lane + 128 * v;
                const float4 bv = col < dv ? *(const float4 *)(sR1 + kk * ldB + col) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    acc6[i][v][0] = fmaf(ar[i], bv.x, acc6[i][v][0]);
                    acc6[i][v][1] = fmaf(ar[i], bv.y, acc6[i][v][1]);
                    acc6[i][v][2] = fmaf(ar[i], bv.z, acc6[i][v][2]);
                    acc6[i][v][3] = fmaf(ar[i], bv.w, acc6[i][v][3]);
                }
            }
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int row = 8 * warp + i;
        if (row >= nr) continue;
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const int col = 4 * lane + 128 * v;
            if (col < dv)
                *(float4 *)(a.sn + ((size_t)(r0 + row) * nh + gh) * dv + col) =
                    make_float4(acc6[i][v][0], acc6[i][v][1], acc6[i][v][2], acc6[i][v][3]);
        }
    }
}

// ------------------------------------------------------------------ near

// Block = (rows, group): 32 query slots = floor(32 / hpg) rows x hpg heads,
// so one staged key/value tile serves every head of the group. 8 warps, 4
// slots each; within a key tile, lane = key. Keys: the window range
// X[lo(r0) .. hi(last row)]; each slot masks to its own row's window.
// Online softmax (running max and sum); the row's window numerator goes to
// `out` and (max, mass, max) to its window header, for the side readout to
// merge.
template <int NV>
__global__ __launch_bounds__(256) void k_near(O1Args a) {
    extern __shared__ float sm[];
    const int dq = a.d + 4, dvq = a.dv + 4;
    float *sQ = sm;
    float *sK = sQ + 32 * dq;
    float *sV = sK + 32 * dq;
    const int g = blockIdx.y;
    const int hpg = a.hpg;
    const int RB = 32 / hpg;
    const int r0 = blockIdx.x * RB;
    const int nr = min(RB, a.R - r0);
    const int nq = nr * hpg;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const O1Meta mt = o1_meta(a, g);
    const int d4 = a.d >> 2, dv4 = a.dv >> 2;

    for (int idx = tid; idx < 32 * d4; idx += 256) {
        const int s = idx / d4, c4 = idx % d4;
        float4 val = make_float4(0.f, 0.f, 0.f, 0.f);
        if (s < nq) {
            const int r = r0 + s / hpg, hh = g * hpg + s % hpg;
            val = ((const float4 *)(a.qr + ((size_t)r * a.nh + hh) * a.d))[c4];
        }
        ((float4 *)(sQ + s * dq))[c4] = val;
    }

    int lo[4], hi[4];
    bool act[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int s = warp * 4 + i;
        act[i] = s < nq;
        const int r = r0 + (act[i] ? s / hpg : 0);
        lo[i] = max(0, mt.len0 + r + 1 - mt.wg);
        hi[i] = mt.len0 + r;
    }
    float mrow[4], lrow[4], acc[4][NV][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        mrow[i] = -INFINITY;
        lrow[i] = 0.f;
#pragma unroll
        for (int v = 0; v < NV; ++v) acc[i][v][0] = acc[i][v][1] = acc[i][v][2] = acc[i][v][3] = 0.f;
    }

    const int xlo = max(0, mt.len0 + r0 + 1 - mt.wg);
    const int xhi = mt.len0 + r0 + nr - 1;
    const int nkeys = xhi - xlo + 1;

    for (int kb = 0; kb < nkeys; kb += 32) {
        const int cnt = min(32, nkeys - kb);
        __syncthreads();
        for (int idx = tid; idx < 32 * d4; idx += 256) {
            const int kk = idx / d4, c4 = idx % d4;
            float4 val = make_float4(0.f, 0.f, 0.f, 0.f);
            if (kk < cnt) val = ((const float4 *)o1_key(a, g, xlo + kb + kk, mt))[c4];
            ((float4 *)(sK + kk * dq))[c4] = val;
        }
        for (int idx = tid; idx < 32 * dv4; idx += 256) {
            const int kk = idx / dv4, c4 = idx % dv4;
            float4 val = make_float4(0.f, 0.f, 0.f, 0.f);
            if (kk < cnt) val = ((const float4 *)o1_val(a, g, xlo + kb + kk, mt))[c4];
            ((float4 *)(sV + kk * dvq))[c4] = val;
        }
        __syncthreads();

        float sc[4] = {0.f, 0.f, 0.f, 0.f};
        const float4 *kp = (const float4 *)(sK + lane * dq);
#pragma unroll 4
        for (int c4 = 0; c4 < d4; ++c4) {
            const float4 kv = kp[c4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float4 qv = ((const float4 *)(sQ + (warp * 4 + i) * dq))[c4];
                sc[i] = fmaf(qv.x, kv.x, sc[i]);
                sc[i] = fmaf(qv.y, kv.y, sc[i]);
                sc[i] = fmaf(qv.z, kv.z, sc[i]);
                sc[i] = fmaf(qv.w, kv.w, sc[i]);
            }
        }
        const int x = xlo + kb + lane;
        float p[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const bool ok = act[i] && lane < cnt && x >= lo[i] && x <= hi[i];
            const float s = ok ? sc[i] * a.scale : -INFINITY;
            const float tm = warp_max(s);
            p[i] = 0.f;
            if (tm == -INFINITY) continue;
            const float mn = fmaxf(mrow[i], tm);
            const float al = expf(mrow[i] - mn);
            p[i] = ok ? expf(s - mn) : 0.f;
            lrow[i] = lrow[i] * al + warp_sum(p[i]);
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                acc[i][v][0] *= al;
                acc[i][v][1] *= al;
                acc[i][v][2] *= al;
                acc[i][v][3] *= al;
            }
            mrow[i] = mn;
        }
        for (int kk = 0; kk < cnt; ++kk) {
            float pk[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) pk[i] = __shfl_sync(0xffffffffu, p[i], kk);
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                const int col = lane * 4 + 128 * v;
                if (col < a.dv) {
                    const float4 vv = *(const float4 *)(sV + kk * dvq + col);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        acc[i][v][0] = fmaf(pk[i], vv.x, acc[i][v][0]);
                        acc[i][v][1] = fmaf(pk[i], vv.y, acc[i][v][1]);
                        acc[i][v][2] = fmaf(pk[i], vv.z, acc[i][v][2]);
                        acc[i][v][3] = fmaf(pk[i], vv.w, acc[i][v][3]);
                    }
                }
            }
        }
    }

    // the window part of the row: numerator into `out`, (reference, mass,
    // max) into the row's window header; the side readout merges
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if (!act[i]) continue;
        const int s = warp * 4 + i;
        const int r = r0 + s / hpg, hh = g * hpg + s % hpg;
        float *o = a.out + ((size_t)r * a.nh + hh) * a.dv;
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const int col = lane * 4 + 128 * v;
            if (col < a.dv) *(float4 *)(o + col) = make_float4(acc[i][v][0], acc[i][v][1], acc[i][v][2], acc[i][v][3]);
        }
        if (lane == 0)
            *(float4 *)(a.fh + ((size_t)r * a.nh + hh) * 4) = make_float4(mrow[i], lrow[i], mrow[i], 0.f);
    }
}

// ----------------------------------------------------------------- merge

// One warp per (row, head): the window part (numerator in `out` relative to
// the reference c_w; header (c_w, mass, true max)) and the side part
// (numerator in sn relative to c_s; header (c_s, mass)) under one exponent
// c = max(true window max, c_s) — the pages' c_all — the denominator floored
// at 1e-30 in those units (o1b_attend), then the gate (dory_gate1).
__global__ __launch_bounds__(256) void k_merge(O1Args a) {
    const int lane = threadIdx.x & 31;
    const size_t rh = (size_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (rh >= (size_t)a.R * a.nh) return;
    const float4 wh = *(const float4 *)(a.fh + rh * 4), sh = *(const float4 *)(a.sh + rh * 4);
    const float cc = fmaxf(wh.z, sh.x);
    const float al = expf(wh.x - cc);
    const float be = sh.x > -INFINITY ? expf(sh.x - cc) : 0.f;
    const float den = fmaxf(al * wh.y + be * sh.y, 1e-30f);
    const float fa = al / den, fb = be / den;
    const int dv4 = a.dv >> 2;
    float4 ow[2], sw[2], gv[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int c4 = lane + 32 * u;
        if (c4 < dv4) {
            ow[u] = ((const float4 *)(a.out + rh * a.dv))[c4];
            sw[u] = ((const float4 *)(a.sn + rh * a.dv))[c4];
            gv[u] = a.gate ? ((const float4 *)(a.gate + rh * a.dv))[c4] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int c4 = lane + 32 * u;
        if (c4 >= dv4) continue;
        float y0 = fa * ow[u].x + fb * sw[u].x, y1 = fa * ow[u].y + fb * sw[u].y;
        float y2 = fa * ow[u].z + fb * sw[u].z, y3 = fa * ow[u].w + fb * sw[u].w;
        if (a.gate) {
            y0 = y0 / (1.f + expf(-gv[u].x));
            y1 = y1 / (1.f + expf(-gv[u].y));
            y2 = y2 / (1.f + expf(-gv[u].z));
            y3 = y3 / (1.f + expf(-gv[u].w));
        }
        ((float4 *)(a.out + rh * a.dv))[c4] = make_float4(y0, y1, y2, y3);
    }
}

// --------------------------------------------------------------- commit

// The pass's rotated keys and values into the ring (o1b_ring_commit: row j
// to slot (head0 + len0 + j) % wg), only the last wg rows since earlier ones
// would be overwritten within the pass; then, by the last block to arrive
// (an atomic ticket, no waiting), every group's meta after R pushes
// (o1b_meta) and the position.
__global__ __launch_bounds__(256) void k_commit(O1Args a) {
    const int g = blockIdx.y;
    const O1Meta mt = o1_meta(a, g);
    const int rstart = max(0, a.R - mt.wg);
    const int d4 = a.d >> 2, dv4 = a.dv >> 2;
    constexpr int RPB = 4;   // rows per block, all loaded before any store
    const int rb = rstart + blockIdx.x * RPB;
    for (int c4 = threadIdx.x; c4 < max(d4, dv4); c4 += blockDim.x) {
        float4 kv[RPB], vv[RPB];
#pragma unroll
        for (int i = 0; i < RPB; ++i) {
            const int r = rb + i;
            const bool in = r < a.R;
            kv[i] = (in && c4 < d4) ? ((const float4 *)(a.kr + ((size_t)r * a.G + g) * a.d))[c4]
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
            vv[i] = (in && c4 < dv4) ? ((const float4 *)(a.v + ((size_t)r * a.G + g) * a.dv))[c4]
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int i = 0; i < RPB; ++i) {
            const int r = rb + i;
            if (r >= a.R) break;
            const int slot = (int)(((long long)mt.head0 + mt.len0 + r) % mt.wg);
            if (c4 < d4) ((float4 *)(a.ring_k + ((size_t)g * a.w + slot) * a.d))[c4] = kv[i];
            if (c4 < dv4) ((float4 *)(a.ring_v + ((size_t)g * a.w + slot) * a.dv))[c4] = vv[i];
        }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const unsigned total = gridDim.x * gridDim.y;
        const unsigned t = atomicAdd(&a.hdr->ticket, 1u);
        if (t == total - 1) {
            __threadfence();
            for (int gg = 0; gg < a.G; ++gg) {
                const long long len0 = a.meta[gg * 4 + 0], head0 = a.meta[gg * 4 + 1];
                const long long wg = a.meta[gg * 4 + 3];
                const long long tot = len0 + a.R;
                if (tot <= wg) {
                    a.meta[gg * 4 + 0] = (uint32_t)tot;
                } else {
                    const long long ev = tot - wg;
                    a.meta[gg * 4 + 0] = (uint32_t)wg;
                    a.meta[gg * 4 + 1] = (uint32_t)((head0 + ev) % wg);
                    a.meta[gg * 4 + 2] = a.meta[gg * 4 + 2] + (uint32_t)ev;
                }
            }
            a.hdr->pos += a.R;
            a.hdr->ticket = 0u;
        }
    }
}

// ------------------------------------------------------------- launchers

extern const char *const o1_stage_names[O1_NUM_STAGES] = {
    "rope", "far_logits", "far_scan", "far_dT", "far_tscan", "side_readout", "gather_tc", "near", "merge", "commit"};

static size_t readout_smem(const O1Args &a) {
    size_t off[6];
    side_layout(a, off);
    return off[5] * sizeof(float);
}

static size_t near_smem(const O1Args &a) { return (size_t)(32 * (a.d + 4) * 2 + 32 * (a.dv + 4)) * sizeof(float); }

namespace {

// A second stream and two events per host thread and device: the far-field
// chain and the window run concurrently after the rotation (they share no
// data), joined before the merge. Fork and join are event record / wait
// pairs, so a capture of the caller's stream captures both branches.
struct O1Aux {
    cudaStream_t st = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};

cudaError_t o1_aux(O1Aux **out) {
    static thread_local O1Aux aux[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    O1Aux &x = aux[dev];
    if (!x.st) {
        // the far branch is the longer one: its blocks go first when SMs free up
        int lo = 0, hi = 0;
        if ((e = cudaDeviceGetStreamPriorityRange(&lo, &hi)) != cudaSuccess) return e;
        if ((e = cudaStreamCreateWithPriority(&x.st, cudaStreamNonBlocking, hi)) != cudaSuccess) return e;
        if ((e = cudaEventCreateWithFlags(&x.fork, cudaEventDisableTiming)) != cudaSuccess) return e;
        if ((e = cudaEventCreateWithFlags(&x.join, cudaEventDisableTiming)) != cudaSuccess) return e;
    }
    *out = &x;
    return cudaSuccess;
}

}  // namespace

// Stages: rope | far_logits, far_scan, far_dT, far_tscan, side_readout |
// gather_tc, near | merge, commit. The two middle branches run concurrently,
// the far one on the library's second stream. With `ev`, events 2i and 2i + 1
// are recorded just before and just after stage i on the stream it runs on.
cudaError_t o1_launch_pass(const O1Args &a, cudaStream_t st, cudaEvent_t const *ev) {
    static bool attrs_set = false;
    if (!attrs_set) {
        cudaFuncSetAttribute(k_side_readout<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        cudaFuncSetAttribute(k_side_readout<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        cudaFuncSetAttribute(k_near<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        cudaFuncSetAttribute(k_near<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        attrs_set = true;
    }
    const int R = a.R;
    const int nblk = (R + O1_SUB - 1) / O1_SUB;
    auto begin = [&](int i, cudaStream_t s) {
        if (ev) cudaEventRecord(ev[2 * i], s);
    };
    auto end = [&](int i, cudaStream_t s) {
        if (ev) cudaEventRecord(ev[2 * i + 1], s);
    };
    O1Aux *aux = nullptr;
    cudaError_t e = o1_aux(&aux);
    if (e != cudaSuccess) return e;
    const cudaStream_t sf = aux->st;   // the far-field branch
    begin(0, st);
    k_rope<<<R, 128, 0, st>>>(a);
    end(0, st);
    cudaEventRecord(aux->fork, st);
    cudaStreamWaitEvent(sf, aux->fork, 0);
    begin(1, sf);
    k_far_logits<<<dim3(nblk, a.nh), 256, 0, sf>>>(a);
    end(1, sf);
    begin(2, sf);
    k_far_scan<<<(a.nh * a.m * 32 + 255) / 256, 256, 0, sf>>>(a);
    end(2, sf);
    begin(3, sf);
    k_far_dT<<<dim3(nblk, a.nh, (a.dv + 63) / 64), 256, 0, sf>>>(a);
    end(3, sf);
    begin(4, sf);
    const size_t n = (size_t)a.nh * a.m * a.dv;
    k_far_tscan<<<(unsigned)((n + 255) / 256), 256, 0, sf>>>(a);
    end(4, sf);
    begin(5, sf);
    if (a.dv <= 128) k_side_readout<1><<<dim3(nblk, a.nh), 256, readout_smem(a), sf>>>(a);
    else k_side_readout<2><<<dim3(nblk, a.nh), 256, readout_smem(a), sf>>>(a);
    end(5, sf);
    cudaEventRecord(aux->join, sf);
    begin(6, st);
    if (a.tc) e = o1_launch_gather_tc(a, st);
    end(6, st);
    begin(7, st);
    if (e == cudaSuccess) {
        if (a.tc) {
            e = o1_launch_near_tc(a, st);
        } else {
            const int RB = 32 / a.hpg;
            const dim3 gn((R + RB - 1) / RB, a.G);
            if (a.dv <= 128) k_near<1><<<gn, 256, near_smem(a), st>>>(a);
            else k_near<2><<<gn, 256, near_smem(a), st>>>(a);
        }
    }
    end(7, st);
    // the far branch is joined even when the window launch failed, so that a
    // capture of `st` stays well formed
    cudaStreamWaitEvent(st, aux->join, 0);
    if (e != cudaSuccess) return e;
    begin(8, st);
    k_merge<<<(unsigned)(((size_t)R * a.nh + 7) / 8), 256, 0, st>>>(a);
    end(8, st);
    begin(9, st);
    const int live = R < a.w ? R : a.w;
    k_commit<<<dim3((live + 3) / 4, a.G), 64, 0, st>>>(a);
    end(9, st);
    return cudaPeekAtLastError();
}

// Fresh far field and ring: M = -inf, Z = 0, T = 0, ring zeros.
__global__ void k_init_state(O1Args a) {
    const size_t nM = (size_t)a.nh * a.m;
    const size_t nT = nM * a.dv;
    const size_t nK = (size_t)a.G * a.w * a.d, nV = (size_t)a.G * a.w * a.dv;
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < nT + nK + nV + nM; i += stride) {
        if (i < nM) {
            a.M[i] = -INFINITY;
            a.Z[i] = 0.f;
        }
        if (i < nT) a.T[i] = 0.f;
        else if (i < nT + nK) a.ring_k[i - nT] = 0.f;
        else if (i < nT + nK + nV) a.ring_v[i - nT - nK] = 0.f;
    }
}

cudaError_t o1_launch_init(const O1Args &a, cudaStream_t st) {
    k_init_state<<<304, 256, 0, st>>>(a);
    return cudaPeekAtLastError();
}
