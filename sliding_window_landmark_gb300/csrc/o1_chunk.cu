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
//  2. k_far_block    per 64-row block: l = scale qt_b . k_e for the keys the
//                    block evicts, the block-local max, E = exp(l - max),
//                    its prefix over rows and total, and the block's value
//                    sum increment sum_j E_bj v_ev(j) (o1b_far_e's dot,
//                    max and prefix; o1b_far_commit's sum; all blocks at once)
//  3. k_far_tscan    the running far max M_c, rescale R_c, mass Z and value
//                    sum T across the blocks (o1b_far_e's rescale and
//                    o1b_far_commit's recurrence T <- R T + dT, as a scan)
//  4. k_side_readout per row: the sinks and the far field (landmark scores,
//                    u = e^{f-F} mu, gains, far mass and numerator) under one
//                    exponent (o1b_attend's sink and far parts)
//  5. k_gather_tc    (tensor-core geometries) the window key sequence as
//                    fp16 hi / lo panels (o1_near_tc.cu)
//  6. k_near_tc      the sliding window on the tensor cores (o1b_attend's
//     or k_near      window part); k_near is the fp32 version for the other
//                    geometries
//  7. k_merge        window and side parts under one exponent, the 1e-30
//                    floor, the gate (o1b_attend's normalisation; dory_gate1)
//  8. k_commit       ring rows and meta (o1b_ring_commit, o1b_meta)
// Stages 2-4 and 5-6 share no data; they run on two streams.
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
    if (a.chain_early) o1_chain_release();
    const int r = blockIdx.x;
    const int half = a.d >> 1;
    const int64_t p = a.hdr->pos + r;
    for (int j = threadIdx.x; j < half; j += blockDim.x) {
        float c = 1.f, s = 0.f;
        if (a.rotate) o1_rope_cs(a.hdr->inv_freq[j], p, c, s);
        // 8 heads' loads ahead of their stores (no queries in a commit pass)
        for (int h0 = 0; a.q && h0 < a.nh; h0 += 8) {
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

// 16-byte asynchronous global -> shared copies (zero-filled when !valid; src
// must still be a valid address then), committed as groups so that the next
// chunk lands while the current one is computed on.
__device__ __forceinline__ void cp_async16(float *dst, const float *src, bool valid) {
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(s), "l"(src), "r"(valid ? 16 : 0) : "memory");
}
__device__ __forceinline__ void cp_async4(float *dst, const float *src) {
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(dst);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(s), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// c[i][j] += a_i . b_j over four k (both operands k-contiguous float4s),
// for the first NI row groups and NJ column groups
template <int NI, int NJ>
__device__ __forceinline__ void fma_k4(float (&c)[4][4], const float4 (&av)[4], const float4 (&bv)[4]) {
#pragma unroll
    for (int i = 0; i < NI; ++i)
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            c[i][j] = fmaf(av[i].x, bv[j].x, c[i][j]);
            c[i][j] = fmaf(av[i].y, bv[j].y, c[i][j]);
            c[i][j] = fmaf(av[i].z, bv[j].z, c[i][j]);
            c[i][j] = fmaf(av[i].w, bv[j].w, c[i][j]);
        }
}
__device__ __forceinline__ void fma4x4_k4(float (&c)[4][4], const float4 (&av)[4], const float4 (&bv)[4]) {
    fma_k4<4, 4>(c, av, bv);
}

// ------------------------------------------------------------- far field

// Per (block c of O1_SUB rows, head): the far logits of the keys the block's
// rows evict (row r >= j0 evicts X[r - j0]), l_bj = scale qt_b . k_ev(j); per
// landmark the block-local max m_b = max_j l_bj, E_bj = e^{l_bj - m_b} with
// its in-block prefix over the rows and its total s_b; and the block's value
// sum increment dT_b = sum_j E_bj v_ev(j), also relative to m_b. The block
// partials compose associatively: k_far_tscan moves them to the running max.
// E and the prefix are 0 on rows that evict nothing.
//
// Layout (256 threads): the logits as two 128-thread halves, each over half
// of every 32-wide k chunk, 4 x 4 register tiles (landmarks x keys) with
// float4 k steps, the halves summed per landmark; the increment with E held
// k-major (a warp's 4 landmarks are one broadcast float4 per key) against
// float4 value columns, NV x 128 columns per warp.
constexpr int FB_LDK = 36;   // 32-wide k chunk + 4
constexpr int FB_LDE = 68;   // E^T row stride (64 landmarks + 4)

__host__ __device__ inline size_t far_block_smem_floats() {
    return (size_t)4 * 64 * FB_LDK + 64 * 65 + 64 * FB_LDE;
}

template <int NV>
__global__ __launch_bounds__(256) void k_far_block(O1Args a) {
    extern __shared__ __align__(16) float sm[];
    o1_chain_wait();
    if (a.chain_early) o1_chain_release();
    const int c = blockIdx.x, gh = blockIdx.y, g = gh / a.hpg;
    const O1Meta mt = o1_meta(a, g);
    const int j0 = mt.wg - mt.len0;
    const int r0 = c * O1_SUB, nr = min(O1_SUB, a.R - r0);
    const int jb = min(nr, max(0, j0 - r0));   // first evicting row of the block
    const int m = a.m, d = a.d, dv = a.dv;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const size_t nm = (size_t)a.nh * m;
    // two stages of [landmark chunk [64][FB_LDK] | key chunk [64][FB_LDK]]
    float *sL = sm + 4 * 64 * FB_LDK;      // [64][65] first half's logits
    float *sEt = sL + 64 * 65;             // [64 rows][FB_LDE] E, k-major
    float *sP = sm;                        // [64][65] second half's logits (after the k loop)
                                           // then two stages of [16][dv + 4] values
    const bool any = jb < nr;
    const int nlt = (m + 31) >> 5;
    if (any) {
        const int half = tid >> 7, gy = (tid & 127) >> 4, gx = tid & 15;
        float acc[2][4][4];
        blk_zero(acc[0]);
        blk_zero(acc[1]);
        auto stage = [&](int kc, float *buf) {
            for (int idx = tid; idx < 2 * 64 * 8; idx += 256) {
                const int which = idx >> 9, row = (idx >> 3) & 63, k = kc + 4 * (idx & 7);
                const float *src = a.qt;
                bool ok = false;
                if (k < d) {
                    if (which == 0) {
                        if (row < m) {
                            src = a.qt + ((size_t)gh * m + row) * d + k;
                            ok = true;
                        }
                    } else if (row >= jb && row < nr) {
                        src = o1_key(a, g, r0 + row - j0, mt) + k;
                        ok = true;
                    }
                }
                cp_async16(buf + which * 64 * FB_LDK + row * FB_LDK + 4 * (idx & 7), src, ok);
            }
            cp_async_commit();
        };
        stage(0, sm);
        for (int kc = 0, it = 0; kc < d; kc += 32, ++it) {
            if (kc + 32 < d) {
                stage(kc + 32, sm + ((it + 1) & 1) * 2 * 64 * FB_LDK);
                cp_async_wait<1>();
            } else {
                cp_async_wait<0>();
            }
            __syncthreads();
            const float *sA = sm + (it & 1) * 2 * 64 * FB_LDK, *sB = sA + 64 * FB_LDK;
#pragma unroll
            for (int s4 = 0; s4 < 4; ++s4) {
                const int ko = 16 * half + 4 * s4;
                float4 av[4], bv[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) bv[j] = *(const float4 *)(sB + (gx + 16 * j) * FB_LDK + ko);
#pragma unroll
                for (int lt = 0; lt < 2; ++lt) {
                    if (lt < nlt) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) av[i] = *(const float4 *)(sA + (32 * lt + gy + 8 * i) * FB_LDK + ko);
                        fma4x4_k4(acc[lt], av, bv);
                    }
                }
            }
            __syncthreads();
        }
        float *dst = half ? sP : sL;
#pragma unroll
        for (int lt = 0; lt < 2; ++lt)
            if (lt < nlt)
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) dst[(32 * lt + gy + 8 * i) * 65 + gx + 16 * j] = acc[lt][i][j];
    }
    __syncthreads();
    // one warp per landmark: max, E, prefix over the block's rows (lane, lane + 32)
    for (int b = warp; b < m; b += 8) {
        const size_t wid = (size_t)gh * m + b;
        const bool e0 = lane >= jb && lane < nr, e1 = lane + 32 >= jb && lane + 32 < nr;
        const float l0 = e0 ? a.scale * (sL[b * 65 + lane] + sP[b * 65 + lane]) : -INFINITY;
        const float l1 = e1 ? a.scale * (sL[b * 65 + lane + 32] + sP[b * 65 + lane + 32]) : -INFINITY;
        const float mx = warp_max(fmaxf(l0, l1));
        const float x0 = e0 ? expf(l0 - mx) : 0.f, x1 = e1 ? expf(l1 - mx) : 0.f;
        float p0 = x0, p1 = x1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float t0 = __shfl_up_sync(0xffffffffu, p0, o), t1 = __shfl_up_sync(0xffffffffu, p1, o);
            if (lane >= o) {
                p0 += t0;
                p1 += t1;
            }
        }
        p1 += __shfl_sync(0xffffffffu, p0, 31);
        sEt[lane * FB_LDE + b] = x0;
        sEt[(lane + 32) * FB_LDE + b] = x1;
        if (lane < nr) {
            a.E[wid * a.cap + r0 + lane] = x0;
            a.P[wid * a.cap + r0 + lane] = p0;
        }
        if (lane + 32 < nr) {
            a.E[wid * a.cap + r0 + lane + 32] = x1;
            a.P[wid * a.cap + r0 + lane + 32] = p1;
        }
        if (lane == 31) {
            a.Fb[(O1_FB_LMAX * nm + wid) * a.nsub + c] = mx;
            a.Fb[(O1_FB_LSUM * nm + wid) * a.nsub + c] = p1;
        }
        if (c == 0 && lane == 0) {
            // the entering (M, Z, Zlo), which k_far_tscan reads while it replaces the state's
            a.Fb[O1_FB_PLANES * nm * a.nsub + wid] = a.M[wid];
            a.Fb[O1_FB_PLANES * nm * a.nsub + nm + wid] = a.Z[wid];
            a.Fb[O1_FB_PLANES * nm * a.nsub + 2 * nm + wid] = a.Zlo[wid];
        }
    }
    if (!any) return;   // k_far_tscan adds no increment for a block without evictions
    __syncthreads();
    // dT[b][t] for the warp's landmarks b = 32 s + 4 warp + (0..3), columns
    // t = 4 lane + 128 v + (0..3)
    float *dst = a.Tp + ((size_t)c * a.nh + gh) * m * dv;
    const int ldv = dv + 4, dv4 = dv >> 2;
    auto stage_v = [&](int k0, float *buf) {
        for (int idx = tid; idx < 16 * dv4; idx += 256) {
            const int kk = idx / dv4, c4 = idx - kk * dv4, jj = k0 + kk;
            const bool ok = jj >= jb && jj < nr;
            cp_async16(buf + kk * ldv + 4 * c4, ok ? o1_val(a, g, r0 + jj - j0, mt) + 4 * c4 : a.qt, ok);
        }
        cp_async_commit();
    };
    for (int s = 0; s < nlt; ++s) {
        float acc[4][NV][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int v = 0; v < NV; ++v) acc[i][v][0] = acc[i][v][1] = acc[i][v][2] = acc[i][v][3] = 0.f;
        stage_v(0, sm);
        for (int k0 = 0, it = 0; k0 < 64; k0 += 16, ++it) {
            if (k0 + 16 < 64) {
                stage_v(k0 + 16, sm + ((it + 1) & 1) * 16 * ldv);
                cp_async_wait<1>();
            } else {
                cp_async_wait<0>();
            }
            __syncthreads();
            const float *sV = sm + (it & 1) * 16 * ldv;
#pragma unroll 4
            for (int kk = 0; kk < 16; ++kk) {
                const float4 e4 = *(const float4 *)(sEt + (k0 + kk) * FB_LDE + 32 * s + 4 * warp);
                const float er[4] = {e4.x, e4.y, e4.z, e4.w};
#pragma unroll
                for (int v = 0; v < NV; ++v) {
                    const int col = 4 * lane + 128 * v;
                    const float4 bv = col < dv ? *(const float4 *)(sV + kk * ldv + col) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        acc[i][v][0] = fmaf(er[i], bv.x, acc[i][v][0]);
                        acc[i][v][1] = fmaf(er[i], bv.y, acc[i][v][1]);
                        acc[i][v][2] = fmaf(er[i], bv.z, acc[i][v][2]);
                        acc[i][v][3] = fmaf(er[i], bv.w, acc[i][v][3]);
                    }
                }
            }
            __syncthreads();
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int b = 32 * s + 4 * warp + i;
            if (b >= m) continue;
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                const int col = 4 * lane + 128 * v;
                if (col < dv)
                    *(float4 *)(dst + (size_t)b * dv + col) =
                        make_float4(acc[i][v][0], acc[i][v][1], acc[i][v][2], acc[i][v][3]);
            }
        }
    }
}

// One thread per (head, landmark, value column), sequential over the pass's
// blocks. With block max m_c and mass s_c from k_far_block: the running far
// max M_c = max(M_{c-1}, m_c), the rescale R_c = e^{M_{c-1} - M_c} (1 when
// the max stays, so an empty field stays empty) and the block factor
// f_c = e^{m_c - M_c} (0 for a block without evictions). The value sum
// entering block c, R_c T_{c-1}, goes to Tp[c] and T_c = R_c T_{c-1} + f_c dT_c.
// Column 0's thread also carries the mass, Z_c = R_c Z_{c-1} + f_c s_c, in
// float-float (the state keeps Z as a high and a low f32 part), and records M_c,
// R_c Z_{c-1} (high and low) and f_c for the side readout; the last M, Z, T
// are the new state (o1b_far_e's max / rescale and o1b_far_commit's
// recurrence, taken as a scan over the blocks).
__global__ __launch_bounds__(256, 4) void k_far_tscan(O1Args a) {
    o1_chain_wait();
    if (a.chain_early) o1_chain_release();
    const size_t n = (size_t)a.nh * a.m * a.dv, nm = (size_t)a.nh * a.m;
    const size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= n) return;
    const size_t wid = idx / a.dv;
    const bool col0 = idx - wid * a.dv == 0;
    const float *lmax = a.Fb + (O1_FB_LMAX * nm + wid) * a.nsub;
    const float *lsum = a.Fb + (O1_FB_LSUM * nm + wid) * a.nsub;
    float *Mc = a.Fb + (O1_FB_MC * nm + wid) * a.nsub;
    float *Bc = a.Fb + (O1_FB_BASE * nm + wid) * a.nsub;
    float *Bl = a.Fb + (O1_FB_BASELO * nm + wid) * a.nsub;
    float *Fc = a.Fb + (O1_FB_FAC * nm + wid) * a.nsub;
    const float *enter = a.Fb + O1_FB_PLANES * nm * a.nsub;
    float T = a.T[idx];
    float Mo = enter[wid];
    o1_ff Zo = ff_make(col0 ? enter[nm + wid] : 0.f, col0 ? enter[2 * nm + wid] : 0.f);
    // 8 blocks' loads issued before their stores (the compiler cannot
    // reorder them itself: the stores may alias later loads for all it knows);
    // few enough registers for the scan to sit beside a window CTA
    for (int c0 = 0; c0 < a.nsub; c0 += 8) {
        float lm[8], dT[8], ls[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int c = c0 + i;
            lm[i] = c < a.nsub ? lmax[c] : -INFINITY;
            dT[i] = c < a.nsub ? a.Tp[(size_t)c * n + idx] : 0.f;
            ls[i] = (col0 && c < a.nsub) ? lsum[c] : 0.f;
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int c = c0 + i;
            if (c < a.nsub) {
                const float Mn = fmaxf(Mo, lm[i]);
                const float Rf = Mn == Mo ? 1.f : expf(Mo - Mn);
                const float f = lm[i] == -INFINITY ? 0.f : expf(lm[i] - Mn);
                const float Ts = Rf * T;
                a.Tp[(size_t)c * n + idx] = Ts;
                T = f != 0.f ? fmaf(f, dT[i], Ts) : Ts;
                if (col0) {
                    // the mass in float-float; M_c, R_c Z_{c-1} (high, low)
                    // and f_c for the side readout
                    const o1_ff base = ff_mul_f(Zo, Rf);
                    Mc[c] = Mn;
                    Bc[c] = base.hi;
                    Bl[c] = base.lo;
                    Fc[c] = f;
                    Zo = ff_fma_f(base, f, ls[i]);
                }
                Mo = Mn;
            }
        }
    }
    if (!a.commit) return;   // attend only: the state keeps its far field
    a.T[idx] = T;
    if (col0) {
        a.M[wid] = Mo;
        a.Z[wid] = Zo.hi;
        a.Zlo[wid] = Zo.lo;
    }
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
    // two stages of each: score chunks, then 16-row B6 chunks
    const size_t r1a = (size_t)2 * 64 * SR_LDQ * (1 + nbt), r1b = (size_t)2 * 16 * (a.dv + 4);
    off[0] = 0;                                              // A6 [K6][SR_LDA]
    off[1] = off[0] + (size_t)K6 * SR_LDA;                   // R1: score chunks, then B6 chunks (2 stages)
    off[2] = off[1] + (r1a > r1b ? r1a : r1b);               // sS [64][64 nbt + 1]
    off[3] = off[2] + (size_t)64 * (64 * nbt + 1);           // R3: mu, then E [64][65]
    off[4] = off[3] + 64 * 65;                               // F, M_c, R_c Z_{c-1} (hi), f_c, (lo) [64] each
    off[5] = off[4] + 5 * 64;                                // total (floats)
}


template <int NV>
__global__ __launch_bounds__(256, 2) void k_side_readout(O1Args a) {
    extern __shared__ __align__(16) float sm[];
    o1_chain_wait();
    const int c = blockIdx.x, gh = blockIdx.y, g = gh / a.hpg;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int ty = tid >> 4, tx = tid & 15;
    const O1Meta mt = o1_meta(a, g);
    const int j0 = mt.wg - mt.len0;
    const int r0 = c * O1_SUB, nr = min(O1_SUB, a.R - r0);
    const int m = a.m, d = a.d, dv = a.dv, nh = a.nh, ns = a.ns;
    const bool far_any = !a.exact && mt.farl0 + max(0, r0 + nr - j0) > 0;
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
    float *sMc = sRow + 64;    // M_c, R_c Z_{c-1} (high, low), f_c per landmark
    float *sBc = sRow + 128;
    float *sFc = sRow + 192;
    float *sBl = sRow + 256;
    if (far_any) {   // mu and the block's far records, in flight under the scores
        float *sMu = sR3;   // [m][65]
        for (int idx = tid; idx < m * m; idx += 256) {
            const int aa = idx / m, b = idx % m;
            sMu[aa * 65 + b] = a.mu[((size_t)gh * m + aa) * m + b];
        }
        const size_t nm = (size_t)nh * m;
        for (int b = tid; b < 64; b += 256) {
            const size_t wid = (size_t)gh * m + b;
            sMc[b] = b < m ? a.Fb[(O1_FB_MC * nm + wid) * a.nsub + c] : 0.f;
            sBc[b] = b < m ? a.Fb[(O1_FB_BASE * nm + wid) * a.nsub + c] : 0.f;
            sBl[b] = b < m ? a.Fb[(O1_FB_BASELO * nm + wid) * a.nsub + c] : 0.f;
            sFc[b] = b < m ? a.Fb[(O1_FB_FAC * nm + wid) * a.nsub + c] : 0.f;
        }
    }

    // 1. scores: columns [0, m) landmarks f_a, [m, m + ns) sinks. A block
    //    without far field needs only the few sink columns: a warp per row.
    if (!far_any && ns <= 8) {
        // the sink keys in shared memory; a warp takes 4 rows at a time
        // (rows i0 + 8 rr), their queries loaded together, lanes across d,
        // and one reduce-scatter leaves score (rr, sink s) in lane 8 rr + s
        float *sSk = sR1;   // [ns][d]
        for (int i = tid; i < ns * d; i += 256) sSk[i] = a.sink_k[(size_t)g * ns * d + i];
        __syncthreads();
        for (int i0 = warp; i0 < nr; i0 += 32) {
            float qv[4][O1_MAX_D / 32];
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) {
                const int i = i0 + 8 * rr;
                const float *qrow = a.qr + ((size_t)(r0 + i) * nh + gh) * d;
#pragma unroll
                for (int t = 0; t < O1_MAX_D / 32; ++t)
                    qv[rr][t] = (i < nr && lane + 32 * t < d) ? qrow[lane + 32 * t] : 0.f;
            }
            float x[32];
#pragma unroll
            for (int v = 0; v < 32; ++v) x[v] = 0.f;
#pragma unroll
            for (int s = 0; s < 8; ++s) {
                if (s >= ns) break;
#pragma unroll
                for (int t = 0; t < O1_MAX_D / 32; ++t) {
                    const float kv = lane + 32 * t < d ? sSk[s * d + lane + 32 * t] : 0.f;
#pragma unroll
                    for (int rr = 0; rr < 4; ++rr) x[rr * 8 + s] = fmaf(qv[rr][t], kv, x[rr * 8 + s]);
                }
            }
            warp_reduce_scatter32(x);
            const int rr = lane >> 3, s = lane & 7, i = i0 + 8 * rr;
            if (s < ns && i < nr) sS[i * ldS + m + s] = a.scale * x[0];
        }
    } else {
        // two stages of [query rows [64][SR_LDQ] | landmark and sink rows [64 nbt][SR_LDQ]]
        float acc[2][4][4];
#pragma unroll
        for (int t = 0; t < 2; ++t) blk_zero(acc[t]);
        const int nrow = 64 * (1 + nbt);
        const bool narrow = m + ns <= 48;   // one tile, its last 16 columns unused
        const bool short_blk = nr <= 16;     // rows 16 .. 63 are past the pass
        auto stage = [&](int kc, float *buf) {
            for (int idx = tid; idx < nrow * 8; idx += 256) {
                const int row = idx >> 3, k = kc + 4 * (idx & 7);
                const float *src = a.qr;
                bool ok = false;
                if (k < d) {
                    if (row < 64) {
                        if (row < nr) {
                            src = a.qr + ((size_t)(r0 + row) * nh + gh) * d + k;
                            ok = true;
                        }
                    } else {
                        const int col = row - 64;
                        if (col < m) {
                            if (far_any) {
                                src = a.kt + ((size_t)g * m + col) * d + k;
                                ok = true;
                            }
                        } else if (col < m + ns) {
                            src = a.sink_k + ((size_t)g * ns + col - m) * d + k;
                            ok = true;
                        }
                    }
                }
                cp_async16(buf + row * SR_LDQ + 4 * (idx & 7), src, ok);
            }
            cp_async_commit();
        };
        stage(0, sR1);
        for (int kc = 0, it = 0; kc < d; kc += 32, ++it) {
            if (kc + 32 < d) {
                stage(kc + 32, sR1 + ((it + 1) & 1) * nrow * SR_LDQ);
                cp_async_wait<1>();
            } else {
                cp_async_wait<0>();
            }
            __syncthreads();
            const float *sQc = sR1 + (it & 1) * nrow * SR_LDQ;   // [64][SR_LDQ]
            const float *sBc = sQc + 64 * SR_LDQ;                // [64 nbt][SR_LDQ]
#pragma unroll 2
            for (int k4 = 0; k4 < 8; ++k4) {
                float4 av[4], bv[4];
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    av[i] = (i == 0 || !short_blk) ? *(const float4 *)(sQc + (ty + 16 * i) * SR_LDQ + 4 * k4)
                                                   : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    if (t < nbt) {
                        if (narrow) {
                            // columns 48..63 are padding: three 16-column groups
#pragma unroll
                            for (int j = 0; j < 3; ++j)
                                bv[j] = *(const float4 *)(sBc + (64 * t + tx + 16 * j) * SR_LDQ + 4 * k4);
                            if (short_blk) fma_k4<1, 3>(acc[t], av, bv);
                            else fma_k4<4, 3>(acc[t], av, bv);
                        } else {
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                bv[j] = *(const float4 *)(sBc + (64 * t + tx + 16 * j) * SR_LDQ + 4 * k4);
                            if (short_blk) fma_k4<1, 4>(acc[t], av, bv);
                            else fma_k4<4, 4>(acc[t], av, bv);
                        }
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
    // the block's E and in-block prefix P [m][64] into the score staging
    // (free now), in flight under steps 2 and 3
    float *sEr = sR1, *sPr = sR1 + (size_t)m * 64;
    if (far_any) {
        const int nr4 = (nr + 3) >> 2;
        for (int idx = tid; idx < m * 16; idx += 256) {
            const int b = idx >> 4, q = idx & 15;
            const bool ok = q < nr4;   // a chunk of 4 rows from r0 (within the padded row stride)
            const size_t at = ((size_t)gh * m + b) * a.cap + r0 + 4 * q;
            cp_async16(sEr + b * 64 + 4 * q, ok ? a.E + at : a.E, ok);
            cp_async16(sPr + b * 64 + 4 * q, ok ? a.P + at : a.P, ok);
        }
        cp_async_commit();
        float *sMu = sR3;   // [m][65]
        // 2. F per row and e^{f - F} (columns [0, m))
        for (int i = warp; i < 64; i += 8) {
            const float v0 = lane < m ? sS[i * ldS + lane] : -INFINITY;
            const float v1 = lane + 32 < m ? sS[i * ldS + lane + 32] : -INFINITY;
            const float F = warp_max(fmaxf(v0, v1));
            if (lane == 0) sRow[i] = F;
            if (lane < m) sS[i * ldS + lane] = expf(v0 - F);
            if (lane + 32 < m) sS[i * ldS + lane + 32] = expf(v1 - F);
        }
        cp_async_wait<0>();   // this thread's E and P chunks have landed
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
        // E of this block's evicting rows, moved from the block max to M_c
        float *sE = sR3;   // [m][65]
        for (int idx = tid; idx < m * 64; idx += 256) {
            const int b = idx >> 6, jj = idx & 63;
            const int r = r0 + jj;
            sE[b * 65 + jj] = (jj < nr && r >= j0) ? sFc[b] * sEr[b * 64 + jj] : 0.f;
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
            // far mass P_b(row) = R_c Z_{c-1} + f_c (in-block prefix), and
            // D = sum_b gain_b P_b, in float-float (the terms can cancel to
            // a small fraction of their size)
            auto pmass = [&](int b) -> o1_ff {
                return ff_fma_f(ff_make(sBc[b], sBl[b]), sFc[b], sPr[b * 64 + i]);
            };
            o1_ff Dd = ff_make(0.f, 0.f);
            if (lane < m) {
                const o1_ff p0 = pmass(lane);
                Dd = ff_add(ff_mul_f(p0, g0), Dd);
            }
            if (lane + 32 < m) {
                const o1_ff p1 = pmass(lane + 32);
                Dd = ff_add(ff_mul_f(p1, g1), Dd);
            }
            Dd = warp_sum(Dd);
            have = ff_nonneg(Dd);
            D = Dd.hi + Dd.lo;
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
    auto stage6 = [&](int k0, float *buf) {
        const int kn = min(16, K6 - k0);
        for (int idx = tid; idx < kn * dv4; idx += 256) {
            const int kk = idx / dv4, c4 = idx - kk * dv4, k = k0 + kk;
            const float *src = a.qr;
            bool ok = true;
            if (k < m) {
                src = Tp + (size_t)k * dv + 4 * c4;
            } else if (k < m + 64) {
                const int jj = k - m, r = r0 + jj;
                ok = jj < nr && r >= j0;
                if (ok) src = o1_val(a, g, r - j0, mt) + 4 * c4;
            } else {
                src = sinks_v + (size_t)(k - m - 64) * dv + 4 * c4;
            }
            cp_async16(buf + kk * ldB + 4 * c4, src, ok);
        }
        cp_async_commit();
    };
    if (kbeg < K6) stage6(kbeg, sR1);
    for (int k0 = kbeg, it = 0; k0 < K6; k0 += 16, ++it) {
        const int kn = min(16, K6 - k0);
        if (k0 + 16 < K6) {
            stage6(k0 + 16, sR1 + ((it + 1) & 1) * 16 * ldB);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const float *sB = sR1 + (it & 1) * 16 * ldB;
        // the in-block coefficients of the warp's rows 8 warp .. 8 warp + 7 are
        // zero past row 8 warp + 7 (causal): those k are skipped
        const int kskip0 = m + 8 * warp + 8, kskip1 = m + 64;
        const int kend = 8 * warp < nr ? kn : 0;   // a warp whose rows are all past the pass skips
#pragma unroll 2
        for (int kk = 0; kk < kend; ++kk) {
            if (k0 + kk >= kskip0 && k0 + kk < kskip1) continue;
            const float4 a0 = *(const float4 *)(sA6 + (k0 + kk) * SR_LDA + 8 * warp);
            const float4 a1 = *(const float4 *)(sA6 + (k0 + kk) * SR_LDA + 8 * warp + 4);
            const float ar[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
            for (int v = 0; v < NV; ++v) {
                const int col = 4 * lane + 128 * v;
                const float4 bv = col < dv ? *(const float4 *)(sB + kk * ldB + col) : make_float4(0.f, 0.f, 0.f, 0.f);
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

// ---------------------------------------------------------- short passes

// A pass of at most O1_SHORT_ROWS rows: the far field and the sinks of head
// blockIdx.x in one CTA, in place of the 64-row block kernels (k_far_block,
// k_far_tscan, k_side_readout). The rows are taken as the oracle takes them
// (row r first inserts the key it evicts, o1b_far_e / o1b_far_commit for one
// key, then reads out, o1b_attend's far and sink parts), but only the
// recurrence of M and Z runs row after row:
//   1. every dot product of the pass at once: the insert logits
//      l_rb = scale qt_b . k_e(r), the far scores f_ra = scale q'_r . kt_a and
//      the sink scores (a warp per 4 row vectors and 8 targets);
//   2. one warp runs the recurrence over the rows with M and Z (float-float)
//      in its registers, two landmarks a lane: M' = max(M, l), rho, e,
//      Z = rho Z + e, and keeps each row's M and Z; beside it, per row,
//      F_r = max_a f_ra, e^{f_ra - F_r} and u_rb = sum_a e^{f_ra - F_r} mu[a][b]
//      (rect);
//   3. a warp per row: c_f = max_b (F + M_b), the gains u_b e^{F+M_b-c_f},
//      D = sum_b gain_b Z_b in float-float and its sign, c_s = max(sink max,
//      c_f), the sink weights and the side header (c_s, side mass);
//   4. the value sums T = rho T + e v_e and the side numerator
//      e^{c_f-c_s} sum_b gain_b T_b + sum_x w_x v_x, row after row with no
//      barrier: each thread owns the entries of T of one value column and
//      every P-th landmark, and P neighbouring lanes sum a column's parts
//      by shuffles.
// A commit pass (short_no_readout) only inserts. The far state is written
// back when the pass commits. The value columns are split over gridDim.y
// CTAs a head (short_col_splits, up to 4; 8 measured slower): each repeats
// the scalars (steps 1-3) and takes one slice of T, of the numerators and of
// the evicted and sink values.
// short_col_splits and the shared-memory layout (ShortLayout) are in o1_common.cuh.

__global__ __launch_bounds__(256, 1) void k_side_short(O1Args a) {
    extern __shared__ __align__(16) float sm[];
    o1_chain_wait();
    if (a.chain_early) o1_chain_release();
    const ShortLayout L = short_layout(a);
    const int h = blockIdx.x, g = h / a.hpg, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int m = a.m, d = a.d, ns = a.ns, R = a.R, nh = a.nh;
    const int dvf = a.dv, dv = L.dvs, c0 = blockIdx.y * dv;   // this CTA's value columns
    const bool lead = blockIdx.y == 0;                        // writes the scalars' results
    const O1Meta mt = o1_meta(a, g);
    const int j0 = mt.wg - mt.len0;   // row r evicts X[r - j0] once r >= j0
    const bool far_on = !a.exact, readout = !a.short_no_readout;
    float *skt = sm + L.skt, *sqt = sm + L.sqt, *smu = sm + L.smu, *sT = sm + L.sT;
    float *ssk = sm + L.ssk, *ssv = sm + L.ssv, *sKe = sm + L.sKe, *sVe = sm + L.sVe, *sQ = sm + L.sQ;
    float *sL = sm + L.sL, *sF = sm + L.sF, *sU = sm + L.sU, *sRho = sm + L.sRho, *sE = sm + L.sE;
    float *sMr = sm + L.sMr, *sZh = sm + L.sZh, *sZl = sm + L.sZl;
    float *sS = sm + L.sS, *sRow = sm + L.sRow;
    auto farl_of = [&](int r) { return far_on ? mt.farl0 + max(0, r - j0 + 1) : 0; };

    // the head's operands and state, and every row's evicted pair and query:
    // 16-byte asynchronous copies, all in flight together (rows of d and dv
    // floats are 16-byte multiples)
    const int d4 = d >> 2, dv4 = dv >> 2;
    if (far_on) {
        for (int i = tid; i < m * d4; i += 256) {
            if (readout) cp_async16(skt + 4 * i, a.kt + (size_t)g * m * d + 4 * i, true);
            cp_async16(sqt + 4 * i, a.qt + (size_t)h * m * d + 4 * i, true);
        }
        // a warp per row, lanes across it: T's rows, the evicted keys and values
        for (int b = warp; b < m; b += 8)
            for (int j = lane; j < dv4; j += 32)
                cp_async16(sT + (size_t)b * L.ldT + 4 * j, a.T + ((size_t)h * m + b) * dvf + c0 + 4 * j, true);
        for (int r = max(j0, 0) + warp; r < R; r += 8) {
            const int x = r - j0;
            const float *ve = o1_val(a, g, x, mt) + c0;
            if (a.commit_rotates && x >= mt.len0) {   // one of the pass's own keys, rotated here
                const float *kraw = a.k + ((size_t)(x - mt.len0) * a.G + g) * d;
                for (int j = lane; j < d4; j += 32)
                    *(float4 *)(sKe + (size_t)r * d + 4 * j) = o1_rot_chunk(a, kraw, j, a.hdr->pos + (x - mt.len0));
            } else {
                const float *ke = o1_key(a, g, x, mt);
                for (int j = lane; j < d4; j += 32) cp_async16(sKe + (size_t)r * d + 4 * j, ke + 4 * j, true);
            }
            for (int j = lane; j < dv4; j += 32) cp_async16(sVe + (size_t)r * dv + 4 * j, ve + 4 * j, true);
        }
    }
    if (readout) {
        for (int i = tid; i < ns * d4; i += 256) cp_async16(ssk + 4 * i, a.sink_k + (size_t)g * ns * d + 4 * i, true);
        for (int x = warp; x < ns; x += 8)
            for (int j = lane; j < dv4; j += 32)
                cp_async16(ssv + (size_t)x * dv + 4 * j, a.sink_v + ((size_t)g * ns + x) * dvf + c0 + 4 * j, true);
        for (int r = warp; r < R; r += 8)
            for (int j = lane; j < d4; j += 32)
                cp_async16(sQ + (size_t)r * d + 4 * j, a.qr + ((size_t)r * nh + h) * d + 4 * j, true);
        if (far_on)
            for (int i = tid; i < m * m; i += 256) cp_async4(smu + i, a.mu + (size_t)h * m * m + i);
    }
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();

    // 1. dot products: task (kind, 4 rows, 8 targets); a warp holds the 4
    //    row vectors in registers, lanes across d, and leaves the 32 dots
    //    through one reduce-scatter (lane l: row l / 8, target l % 8)
    {
        const int nc0 = (m + 7) / 8, nc2 = (ns + 7) / 8, per = 2 * nc0 + nc2, nrg = (R + 3) / 4;
        for (int i = warp; i < nrg * per; i += 8) {
            const int rg = i / per, k = i - rg * per, r0 = 4 * rg, rl = min(R, r0 + 4) - 1;
            const float *x, *rows;
            float *out;
            int n0, n;
            if (k < nc0) {   // the insert logits of the keys rows r0.. evict
                if (!far_on || rl < j0) continue;
                x = sKe, rows = sqt, out = sL, n0 = 8 * k, n = m;
            } else if (k < 2 * nc0) {   // the far scores of rows r0..
                if (!readout || farl_of(rl) <= 0) continue;
                x = sQ, rows = skt, out = sF, n0 = 8 * (k - nc0), n = m;
            } else {   // their sink scores
                if (!readout) continue;
                x = sQ, rows = ssk, out = sS, n0 = 8 * (k - 2 * nc0), n = ns;
            }
            float4 xr[4][2];
#pragma unroll
            for (int ri = 0; ri < 4; ++ri)
#pragma unroll
                for (int u = 0; u < 2; ++u)
                    xr[ri][u] = (r0 + ri < R && lane + 32 * u < d4)
                                    ? ((const float4 *)(x + (size_t)(r0 + ri) * d))[lane + 32 * u]
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
            float p[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) p[j] = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (n0 + j < n) {
                    const float4 *rw = (const float4 *)(rows + (size_t)(n0 + j) * d);
#pragma unroll
                    for (int u = 0; u < 2; ++u)
                        if (lane + 32 * u < d4) {
                            const float4 y = rw[lane + 32 * u];
#pragma unroll
                            for (int ri = 0; ri < 4; ++ri) {
                                float &pp = p[8 * ri + j];
                                pp = fmaf(xr[ri][u].x, y.x, pp);
                                pp = fmaf(xr[ri][u].y, y.y, pp);
                                pp = fmaf(xr[ri][u].z, y.z, pp);
                                pp = fmaf(xr[ri][u].w, y.w, pp);
                            }
                        }
                }
            }
            warp_reduce_scatter32(p);
            const int r = r0 + (lane >> 3), b = n0 + (lane & 7);
            if (r < R && b < n) out[(size_t)r * n + b] = a.scale * p[0];
        }
    }
    __syncthreads();

    // 2. warp 0: the recurrence of M and Z (float-float) over the rows in its
    //    registers, landmarks b = lane, lane + 32, each row's rescale and
    //    weight kept for the value sums and its M, Z for its readout.
    //    Warps 1..7 meanwhile, per row with a far field: F, e^{f - F} in
    //    place, u (rect).
    if (warp == 0) {
        if (far_on) {
            float Mr[2];
            o1_ff Zr[2];
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int b = lane + 32 * k;
                Mr[k] = b < m ? a.M[(size_t)h * m + b] : -INFINITY;
                Zr[k] = b < m ? ff_make(a.Z[(size_t)h * m + b], a.Zlo[(size_t)h * m + b]) : ff_make(0.f, 0.f);
            }
            for (int r = 0; r < R; ++r) {
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int b = lane + 32 * k;
                    if (b >= m) continue;
                    if (r >= j0) {   // insert the evicted key
                        const float l = sL[(size_t)r * m + b], Mo = Mr[k];
                        const float Mn = fmaxf(Mo, l);
                        const float rho = (Mn == Mo) ? 1.f : expf(Mo - Mn);
                        const float e = expf(l - Mn);
                        Zr[k] = ff_add_f(ff_mul_f(Zr[k], rho), e);
                        Mr[k] = Mn;
                        sRho[(size_t)r * m + b] = rho;
                        sE[(size_t)r * m + b] = e;
                    }
                    if (readout) {
                        sMr[(size_t)r * m + b] = Mr[k];
                        sZh[(size_t)r * m + b] = Zr[k].hi;
                        sZl[(size_t)r * m + b] = Zr[k].lo;
                    }
                }
            }
            // the new M, Z go to scratch, not to the state: the head's other
            // column-slice CTAs may not have read the old ones yet. The
            // pass's ring push stores them (far_copy).
            if (a.commit && lead) {
                const size_t nm = (size_t)nh * m;
                float *out = a.Fb + (size_t)O1_FB_PLANES * nm * a.nsub;
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int b = lane + 32 * k;
                    if (b < m) {
                        out[(size_t)h * m + b] = Mr[k];
                        out[nm + (size_t)h * m + b] = Zr[k].hi;
                        out[2 * nm + (size_t)h * m + b] = Zr[k].lo;
                    }
                }
            }
        }
    } else if (readout && far_on) {
        for (int r = warp - 1; r < R; r += 7) {
            if (farl_of(r) <= 0) continue;
            float *f = sF + (size_t)r * m;
            const float f0 = lane < m ? f[lane] : -INFINITY, f1 = lane + 32 < m ? f[lane + 32] : -INFINITY;
            const float F = warp_max(fmaxf(f0, f1));
            if (lane < m) f[lane] = expf(f0 - F);
            if (lane + 32 < m) f[lane + 32] = expf(f1 - F);
            if (lane == 0) sRow[4 * r] = F;
            __syncwarp();
            for (int b = lane; b < m; b += 32) {
                float u0 = 0.f, u1 = 0.f;
                int aa = 0;
                for (; aa + 1 < m; aa += 2) {
                    u0 = fmaf(f[aa], smu[aa * m + b], u0);
                    u1 = fmaf(f[aa + 1], smu[(aa + 1) * m + b], u1);
                }
                if (aa < m) u0 = fmaf(f[aa], smu[aa * m + b], u0);
                float u = u0 + u1;
                if (a.rect) u = fmaxf(u, 0.f);
                sU[(size_t)r * m + b] = u;
            }
        }
    }
    __syncthreads();

    // 3. each row's readout scalars, a warp per row: c_f = max_b (F + M_b),
    //    the gains, D and its sign, c_s = max(sink max, c_f), the sink
    //    weights, the side header (c_s, side mass)
    if (readout) {
        for (int r = warp; r < R; r += 8) {
            float cf = -INFINITY;
            bool have = false;
            o1_ff D = ff_make(0.f, 0.f);
            if (farl_of(r) > 0) {
                const float F = sRow[4 * r];
                float c = -INFINITY;
#pragma unroll
                for (int k = 0; k < 2; ++k)
                    if (lane + 32 * k < m) c = fmaxf(c, F + sMr[(size_t)r * m + lane + 32 * k]);
                cf = warp_max(c);
                o1_ff Dp = ff_make(0.f, 0.f);
#pragma unroll
                for (int k = 0; k < 2; ++k) {
                    const int b = lane + 32 * k;
                    if (b < m) {
                        const size_t o = (size_t)r * m + b;
                        const float gn = sU[o] * expf(F + sMr[o] - cf);
                        sU[o] = gn;
                        Dp = ff_add(Dp, ff_mul_f(ff_make(sZh[o], sZl[o]), gn));
                    }
                }
                D = warp_sum(Dp);
                have = ff_nonneg(D);
            }
            const float s0 = lane < ns ? sS[(size_t)r * ns + lane] : -INFINITY;
            const float s1 = lane + 32 < ns ? sS[(size_t)r * ns + lane + 32] : -INFINITY;
            const float cs = fmaxf(warp_max(fmaxf(s0, s1)), cf);
            const float fs = have ? expf(cf - cs) : 0.f;
            const float w0 = lane < ns ? expf(s0 - cs) : 0.f, w1 = lane + 32 < ns ? expf(s1 - cs) : 0.f;
            if (lane < ns) sS[(size_t)r * ns + lane] = w0;
            if (lane + 32 < ns) sS[(size_t)r * ns + lane + 32] = w1;
            const float side = (have ? fs * (D.hi + D.lo) : 0.f) + warp_sum(w0 + w1);
            if (lane == 0) {
                sRow[4 * r + 1] = fs;
                if (lead)
                    *(float4 *)(a.sh + ((size_t)r * nh + h) * 4) =
                        make_float4(cs, cs > -INFINITY ? side : 0.f, 0.f, 0.f);
            }
        }
    }
    __syncthreads();

    // 4. value sums and side numerators, row after row: thread (t, pi) owns
    //    T[b][t] for b = pi, pi + P, ..., eight of them in registers at a time
    const int P = L.P, t = tid / P, pi = tid - t * P;
    const bool act = t < dv;
    float *Tt = sT + (act ? t : 0);
    const int nb = act ? (m - pi + P - 1) / P : 0;   // the thread's landmarks
    for (int r = 0; r < R; ++r) {
        const bool ins = far_on && r >= j0;
        const float fs = readout ? sRow[4 * r + 1] : 0.f;
        float acc = 0.f;
        if (ins || fs != 0.f) {
            const float ve = ins && act ? sVe[(size_t)r * dv + t] : 0.f;
            const float *rho = sRho + (size_t)r * m, *e = sE + (size_t)r * m, *gn = sU + (size_t)r * m;
            for (int j = 0; j < nb; j += 8) {
                float tv[8], rv[8], ev[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int b = pi + (j + u) * P;
                    const bool in = j + u < nb;
                    tv[u] = in ? Tt[(size_t)b * L.ldT] : 0.f;
                    rv[u] = in && ins ? rho[b] : 1.f;
                    ev[u] = in && ins ? e[b] : 0.f;
                }
                if (ins) {
#pragma unroll
                    for (int u = 0; u < 8; ++u) tv[u] = fmaf(rv[u], tv[u], ev[u] * ve);
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        if (j + u < nb) Tt[(size_t)(pi + (j + u) * P) * L.ldT] = tv[u];
                }
                if (fs != 0.f) {
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        if (j + u < nb) acc = fmaf(gn[pi + (j + u) * P], tv[u], acc);
                }
            }
            acc *= fs;
        }
        if (!readout) continue;
        if (act) {
            const float *w = sS + (size_t)r * ns;
            for (int x = pi; x < ns; x += P) acc = fmaf(w[x], ssv[(size_t)x * dv + t], acc);
        }
        for (int o = 1; o < P; o <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (act && pi == 0) a.sn[((size_t)r * nh + h) * dvf + c0 + t] = acc;
    }
    if (a.commit && far_on && act)   // attend only: the state keeps its far field
        for (int b = pi; b < m; b += P) a.T[((size_t)h * m + b) * dvf + c0 + t] = Tt[(size_t)b * L.ldT];
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
    o1_chain_wait();
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

// ------------------------------------------------------- short passes

// Window of a short pass (2 .. O1_SMALL_NQ / hpg rows, e.g. a speculative
// draft): the group's keys X[xlo .. len0 + R - 1] (row 0's window start to
// the last row's own key) split into key slices of KS <= 64, one block per
// (slice, group) for all R x hpg query vectors at once, each a slice-local
// softmax (max, sum, value sums); k_near_small_merge combines the slices.
// The row-block tensor-core kernel would give one CTA per head a whole
// window to walk. Register-tiled: queries and keys k-contiguous in padded
// rows, the 64 x 64 score tile as 4 x 4 per thread over float4 k steps (only
// the query row groups the pass has), P.V as 16 query rows x 4 columns per
// thread. Smem: queries [64][d + 4], keys [64][d + 4], values [64][dv + 4],
// scores [64][65].
constexpr int NS_LD = 65;
static size_t near_small_smem(const O1Args &a, int KS) {
    (void)KS;
    return ((size_t)128 * (a.d + 4) + (size_t)64 * (a.dv + 4) + 64 * NS_LD) * sizeof(float);
}

template <int NI, int NJ>
__device__ __forceinline__ void ns_scores(float (&c)[4][4], const float *sQ, const float *sK, int ld, int d4) {
    const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
#pragma unroll 2
    for (int k4 = 0; k4 < d4; ++k4) {
        float4 av[4], bv[4];
#pragma unroll
        for (int i = 0; i < NI; ++i) av[i] = *(const float4 *)(sQ + (ty + 16 * i) * ld + 4 * k4);
#pragma unroll
        for (int j = 0; j < NJ; ++j) bv[j] = *(const float4 *)(sK + (tx + 16 * j) * ld + 4 * k4);
        fma_k4<NI, NJ>(c, av, bv);
    }
}
// the NJ key tiles of 16 that hold the slice's keys
template <int NI>
__device__ __forceinline__ void ns_scores_j(float (&c)[4][4], const float *sQ, const float *sK, int ld, int d4, int nj) {
    switch (nj) {
        case 1: ns_scores<NI, 1>(c, sQ, sK, ld, d4); break;
        case 2: ns_scores<NI, 2>(c, sQ, sK, ld, d4); break;
        case 3: ns_scores<NI, 3>(c, sQ, sK, ld, d4); break;
        default: ns_scores<NI, 4>(c, sQ, sK, ld, d4); break;
    }
}

__global__ __launch_bounds__(256, 1) void k_near_small(O1Args a, int KS) {
    extern __shared__ __align__(16) float sm[];
    o1_chain_wait();
    if (a.chain_early) o1_chain_release();
    const int s = blockIdx.x, g = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int ty = tid >> 4, tx = tid & 15;
    const O1Meta mt = o1_meta(a, g);
    const int R = a.R, hpg = a.hpg, d = a.d, dv = a.dv, nq = R * hpg;
    const int xlo = max(0, mt.len0 + 1 - mt.wg);   // row 0's first window key
    const int x0 = xlo + s * KS;
    const int cnt = max(0, min(KS, mt.len0 + R - x0));
    const size_t slot = (size_t)g * O1_SMALL_NS + s;
    float *pv = a.Sp + slot * O1_SMALL_NQ * dv;                                          // [nq][dv]
    float *pml = a.Sp + (size_t)a.G * O1_SMALL_NS * O1_SMALL_NQ * dv + slot * O1_SMALL_NQ * 2;   // [nq][2]
    if (cnt == 0) {
        for (int q = tid; q < nq; q += blockDim.x) {
            pml[2 * q] = -INFINITY;
            pml[2 * q + 1] = 0.f;
        }
        return;
    }
    const int ld = d + 4, ldv = dv + 4, d4 = d >> 2, dv4 = dv >> 2;
    const int ngi = (nq + 15) >> 4;   // query row groups of 16 in use
    float *sQ = sm;                   // [64][ld]
    float *sK = sQ + 64 * ld;         // [64][ld]
    float *sV = sK + 64 * ld;         // [64][ldv]
    float *sS = sV + 64 * ldv;        // [64][NS_LD]
    // the pass's rotated queries of this group (query q = row q / hpg, head
    // q % hpg) and the slice's keys and values: a warp per row, 16-byte
    // asynchronous copies across its lanes. The rows past nq and past cnt
    // are not loaded: their scores are never read.
    for (int i = warp; i < nq + 2 * cnt; i += 8) {
        const float *src;
        float *dst;
        int n4;
        if (i < nq) {
            const int r = i / hpg, hh = i - r * hpg;
            src = a.qr + ((size_t)r * a.nh + g * hpg + hh) * d, dst = sQ + i * ld, n4 = d4;
        } else if (i < nq + cnt) {
            src = o1_key(a, g, x0 + i - nq, mt), dst = sK + (i - nq) * ld, n4 = d4;
        } else {
            src = o1_val(a, g, x0 + i - nq - cnt, mt), dst = sV + (i - nq - cnt) * ldv, n4 = dv4;
        }
        for (int c = lane; c < n4; c += 32) cp_async16(dst + 4 * c, src + 4 * c, true);
    }
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();
    // scores, masked to each query row's window, into sS
    {
        float c[4][4];
        blk_zero(c);
        const int nj = (cnt + 15) >> 4;
        switch (ngi) {
            case 1: ns_scores_j<1>(c, sQ, sK, ld, d4, nj); break;
            case 2: ns_scores_j<2>(c, sQ, sK, ld, d4, nj); break;
            case 3: ns_scores_j<3>(c, sQ, sK, ld, d4, nj); break;
            default: ns_scores_j<4>(c, sQ, sK, ld, d4, nj); break;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int q = ty + 16 * i;
            if (i >= ngi || q >= nq) continue;
            const int r = q / hpg;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int key = tx + 16 * j, x = x0 + key;
                // row r's window: X[max(0, len0 + r + 1 - wg) .. len0 + r]
                const bool vis = key < cnt && x <= mt.len0 + r && x >= mt.len0 + r + 1 - mt.wg;
                sS[q * NS_LD + key] = vis ? a.scale * c[i][j] : -INFINITY;
            }
        }
    }
    __syncthreads();
    // slice-local softmax per query vector (one warp each; keys lane, lane + 32)
    for (int q = warp; q < nq; q += 8) {
        const float s0 = sS[q * NS_LD + lane], s1 = sS[q * NS_LD + lane + 32];
        const float mx = warp_max(fmaxf(s0, s1));
        const float e0 = s0 > -INFINITY ? expf(s0 - mx) : 0.f, e1 = s1 > -INFINITY ? expf(s1 - mx) : 0.f;
        sS[q * NS_LD + lane] = e0;
        sS[q * NS_LD + lane + 32] = e1;
        const float l = warp_sum(e0 + e1);
        if (lane == 0) {
            pml[2 * q] = mx;
            pml[2 * q + 1] = l;
        }
    }
    __syncthreads();
    // value sums: thread = (group of 8 query vectors, 4 columns), 32 accumulators
    {
        const int c4 = tid & 63;
        for (int qg = tid >> 6; 8 * qg < nq; qg += 4) {
            if (c4 >= dv4) break;
            float acc[8][4];
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
            for (int key = 0; key < cnt; ++key) {
                const float4 v = *(const float4 *)(sV + key * ldv + 4 * c4);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float w = sS[(8 * qg + i) * NS_LD + key];
                    acc[i][0] = fmaf(w, v.x, acc[i][0]);
                    acc[i][1] = fmaf(w, v.y, acc[i][1]);
                    acc[i][2] = fmaf(w, v.z, acc[i][2]);
                    acc[i][3] = fmaf(w, v.w, acc[i][3]);
                }
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int q = 8 * qg + i;
                if (q < nq)
                    *(float4 *)(pv + (size_t)q * dv + 4 * c4) = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
            }
        }
    }
}

// Combine the key slices of a short pass per (row, head, 64 columns): 256
// threads = 4 slice groups x 64 columns, an online max over the slices, then
// the window numerator into `out` (relative to the window max c_w) and the
// window header (c_w, mass, c_w, 0), as the row-block window kernels write
// them for k_merge.
__global__ __launch_bounds__(256) void k_near_small_merge(O1Args a, int nsl) {
    __shared__ float smx[4][64], sl[4][64], sacc[4][64];
    o1_chain_wait();
    const int rh = blockIdx.x, r = rh / a.nh, gh = rh - r * a.nh, g = gh / a.hpg;
    const int q = r * a.hpg + (gh - g * a.hpg);
    const int tid = threadIdx.x, sg = tid >> 6, col = tid & 63, t = blockIdx.y * 64 + col;
    const float *pvb = a.Sp + (size_t)g * O1_SMALL_NS * O1_SMALL_NQ * a.dv;
    const float *pmb = a.Sp + (size_t)a.G * O1_SMALL_NS * O1_SMALL_NQ * a.dv + (size_t)g * O1_SMALL_NS * O1_SMALL_NQ * 2;
    float mx = -INFINITY, l = 0.f, acc = 0.f;
    for (int c0 = sg; c0 < nsl; c0 += 4 * 8) {
        float mc[8], lc[8], vc[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int c = c0 + 4 * u;
            const bool in = c < nsl;
            const size_t sq = (size_t)c * O1_SMALL_NQ + q;
            mc[u] = in ? pmb[2 * sq] : -INFINITY;
            lc[u] = in ? pmb[2 * sq + 1] : 0.f;
            vc[u] = (in && t < a.dv) ? pvb[sq * a.dv + t] : 0.f;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            if (mc[u] == -INFINITY) continue;
            const float mn = fmaxf(mx, mc[u]);
            const float fo = expf(mx - mn), fc = expf(mc[u] - mn);
            l = l * fo + lc[u] * fc;
            acc = acc * fo + vc[u] * fc;
            mx = mn;
        }
    }
    smx[sg][col] = mx;
    sl[sg][col] = l;
    sacc[sg][col] = acc;
    __syncthreads();
    if (sg == 0) {
        float M = -INFINITY;
#pragma unroll
        for (int u = 0; u < 4; ++u) M = fmaxf(M, smx[u][col]);
        float L = 0.f, A = 0.f;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (smx[u][col] == -INFINITY) continue;
            const float f = expf(smx[u][col] - M);
            L = fmaf(sl[u][col], f, L);
            A = fmaf(sacc[u][col], f, A);
        }
        if (t < a.dv) a.out[((size_t)r * a.nh + gh) * a.dv + t] = A;
        if (blockIdx.y == 0 && col == 0) *(float4 *)(a.fh + ((size_t)r * a.nh + gh) * 4) = make_float4(M, L, M, 0.f);
    }
}

// Host side of the short-pass window: slices of KS keys covering the widest
// window plus the pass, at most O1_SMALL_NS per group and at most 64 keys
// each (windows up to about 4 k keys); 0 when the pass is not short or the
// window too long, and the row-block window kernels take it.
static int near_small_ks(const O1Args &a) {
    if (!a.Sp || a.R < 2 || a.R * a.hpg > O1_SMALL_NQ) return 0;
    const int nx = a.w + a.R - 1;
    int KS = (nx + O1_SMALL_NS - 1) / O1_SMALL_NS;
    KS = KS < 8 ? 8 : (KS + 7) / 8 * 8;
    if (KS > 64 || near_small_smem(a, KS) > 227 * 1024) return 0;   // a slice is one 64-key score tile
    return KS;
}

// ----------------------------------------------------------------- merge

// One warp per (row, head): the window part (numerator in `out` relative to
// the reference c_w; header (c_w, mass, true max)) and the side part
// (numerator in sn relative to c_s; header (c_s, mass)) under one exponent
// c = max(true window max, c_s) — the pages' c_all — the denominator floored
// at 1e-30 in those units (o1b_attend), then the gate (dory_gate1).
// A window split over key ranges (wsplit > 1) adds its other splits'
// numerators and masses, each from its own reference, under the same c.
__device__ void merge_splits(const O1Args &a, size_t rh, float4 wh, float4 sh) {
    const int lane = threadIdx.x & 31, S = a.wsplit, dv4 = a.dv >> 2;
    const size_t RN = (size_t)a.R * a.nh;
    const float *hs = a.wpart + (size_t)(S - 1) * RN * a.dv;   // split headers [S-1][R][nh][4]
    float cc = fmaxf(wh.z, sh.x);
    for (int s = 1; s < S; ++s) cc = fmaxf(cc, hs[((size_t)(s - 1) * RN + rh) * 4 + 2]);
    const float al = wh.x > -INFINITY ? expf(wh.x - cc) : 0.f;
    const float be = sh.x > -INFINITY ? expf(sh.x - cc) : 0.f;
    float den = al * wh.y + be * sh.y;
    float4 acc[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int c4 = lane + 32 * u;
        acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (c4 >= dv4) continue;
        const float4 ow = ((const float4 *)(a.out + rh * a.dv))[c4], sw = ((const float4 *)(a.sn + rh * a.dv))[c4];
        acc[u] = make_float4(al * ow.x + be * sw.x, al * ow.y + be * sw.y, al * ow.z + be * sw.z, al * ow.w + be * sw.w);
    }
    for (int s = 1; s < S; ++s) {
        const float4 h = *(const float4 *)(hs + ((size_t)(s - 1) * RN + rh) * 4);
        if (!(h.x > -INFINITY)) continue;   // no key of this row in that split
        const float f = expf(h.x - cc);
        den += f * h.y;
        const float4 *on = (const float4 *)(a.wpart + ((size_t)(s - 1) * RN + rh) * a.dv);
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const int c4 = lane + 32 * u;
            if (c4 >= dv4) continue;
            const float4 o = on[c4];
            acc[u].x = fmaf(f, o.x, acc[u].x);
            acc[u].y = fmaf(f, o.y, acc[u].y);
            acc[u].z = fmaf(f, o.z, acc[u].z);
            acc[u].w = fmaf(f, o.w, acc[u].w);
        }
    }
    const float rd = 1.f / fmaxf(den, 1e-30f);
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const int c4 = lane + 32 * u;
        if (c4 >= dv4) continue;
        float y[4] = {acc[u].x * rd, acc[u].y * rd, acc[u].z * rd, acc[u].w * rd};
        if (a.gate) {
            const float4 gv = ((const float4 *)(a.gate + rh * a.dv))[c4];
            y[0] = y[0] / (1.f + expf(-gv.x));
            y[1] = y[1] / (1.f + expf(-gv.y));
            y[2] = y[2] / (1.f + expf(-gv.z));
            y[3] = y[3] / (1.f + expf(-gv.w));
        }
        ((float4 *)(a.out + rh * a.dv))[c4] = make_float4(y[0], y[1], y[2], y[3]);
    }
}

__global__ __launch_bounds__(256) void k_merge(O1Args a) {
    const int lane = threadIdx.x & 31;
    const size_t rh = (size_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (rh >= (size_t)a.R * a.nh) return;
    const float4 wh = *(const float4 *)(a.fh + rh * 4), sh = *(const float4 *)(a.sh + rh * 4);
    if (a.wsplit > 1) {
        merge_splits(a, rh, wh, sh);
        return;
    }
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

// Every block of a ring push arrives once its rows are written; the last to
// arrive (an atomic ticket, no waiting) advances every group's meta by R
// pushes (o1b_meta) and the position. After a short far kernel (far_copy)
// block (0, 0) first stores the new M, Z, Zlo it left in scratch.
__device__ __forceinline__ void commit_meta(const O1Args &a) {
    if (a.far_copy && blockIdx.x == 0 && blockIdx.y == 0) {
        const size_t nm = (size_t)a.nh * a.m;
        const float *src = a.Fb + (size_t)O1_FB_PLANES * nm * a.nsub;
        for (size_t i = threadIdx.x; i < nm; i += blockDim.x) {
            a.M[i] = src[i];
            a.Z[i] = src[nm + i];
            a.Zlo[i] = src[2 * nm + i];
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

// The pass's rotated keys and values into the ring (o1b_ring_commit: row j
// to slot (head0 + len0 + j) % wg), only the last wg rows since earlier ones
// would be overwritten within the pass; then, by the last block to arrive
// (an atomic ticket, no waiting), every group's meta after R pushes
// (o1b_meta) and the position.
__global__ __launch_bounds__(256) void k_commit(O1Args a) {
    o1_chain_wait();   // ends a pass: releases nothing early
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
    commit_meta(a);
}

// The ring push of a short commit pass that runs without the rotation
// kernel: block (row, group), thread j rotates pair (j, j + d/2) of the row's
// raw key to its position as k_rope does and writes it, with the value, to
// the row's ring slot; then the meta and position as k_commit.
__global__ __launch_bounds__(128) void k_commit_rot(O1Args a) {
    o1_chain_wait();   // ends a pass: releases nothing early
    const int g = blockIdx.y;
    const O1Meta mt = o1_meta(a, g);
    const int r = max(0, a.R - mt.wg) + (int)blockIdx.x;
    if (r < a.R) {
        const int slot = (int)(((long long)mt.head0 + mt.len0 + r) % mt.wg);
        const float *kraw = a.k + ((size_t)r * a.G + g) * a.d;
        float *rk = a.ring_k + ((size_t)g * a.w + slot) * a.d;
        const int half = a.d >> 1;
        const long long p = a.hdr->pos + r;
        for (int j = threadIdx.x; j < half; j += blockDim.x) {
            float c = 1.f, s = 0.f;
            if (a.rotate) o1_rope_cs(a.hdr->inv_freq[j], p, c, s);
            const float x0 = kraw[j], x1 = kraw[j + half];
            rk[j] = x0 * c - x1 * s;
            rk[j + half] = x1 * c + x0 * s;
        }
        const float4 *vs = (const float4 *)(a.v + ((size_t)r * a.G + g) * a.dv);
        float4 *vd = (float4 *)(a.ring_v + ((size_t)g * a.w + slot) * a.dv);
        for (int c4 = threadIdx.x; c4 < (a.dv >> 2); c4 += blockDim.x) vd[c4] = vs[c4];
    }
    commit_meta(a);
}

// ------------------------------------------------------------- launchers

extern const char *const o1_stage_names[O1_NUM_STAGES] = {
    "rope", "far_block", "far_tscan", "side_readout", "gather_tc", "near", "merge", "commit"};

static size_t readout_smem(const O1Args &a) {
    size_t off[6];
    side_layout(a, off);
    return off[5] * sizeof(float);
}

static size_t near_smem(const O1Args &a) { return (size_t)(32 * (a.d + 4) * 2 + 32 * (a.dv + 4)) * sizeof(float); }

// Dynamic shared memory above 48 KB for the kernels that take it, set once
// per device.
static void chunk_attrs() {
    static unsigned long long done = 0;
    unsigned long long bit = 0;
    if (!o1_attrs_needed(&done, &bit)) return;
    cudaFuncSetAttribute(k_side_readout<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    cudaFuncSetAttribute(k_side_readout<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    cudaFuncSetAttribute(k_far_block<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, 96 * 1024);
    cudaFuncSetAttribute(k_far_block<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, 96 * 1024);
    cudaFuncSetAttribute(k_near_small, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    cudaFuncSetAttribute(k_side_short, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    cudaFuncSetAttribute(k_near<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    cudaFuncSetAttribute(k_near<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    o1_attrs_done(&done, bit);
}

namespace {

// A second stream and two events per host thread and device: the far-field
// chain and the window run concurrently after the rotation (they share no
// data), joined before the merge. Fork and join are event record / wait
// pairs, so a capture of the caller's stream captures both branches.
struct O1Aux {
    cudaStream_t st = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
    // Released when the host thread exits, so that short-lived or pooled
    // threads leave nothing behind. (Should the runtime already be unloading,
    // these calls return an error and change nothing.)
    ~O1Aux() {
        if (join) cudaEventDestroy(join);
        if (fork) cudaEventDestroy(fork);
        if (st) cudaStreamDestroy(st);
    }
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

// Stages: rope | far_block, far_tscan, side_readout | gather_tc, near |
// merge, commit. The two middle branches run concurrently,
// the far one on the library's second stream. With `ev`, events 2i and 2i + 1
// are recorded just before and just after stage i on the stream it runs on.
cudaError_t o1_launch_pass(const O1Args &a_in, cudaStream_t st, cudaEvent_t const *ev) {
    chunk_attrs();
    O1Args a = a_in;
    const int R = a.R;
    const int KS = near_small_ks(a);   // > 0: a short pass, its window split over key slices
    if (KS) a.tc = 0;
    // a short pass's window kernels are scheduled under their predecessors'
    // ends (its CTAs fit beside the far branch's few)
    if (KS && R <= O1_SHORT_ROWS) a.chain_early = 1;
    {
        // window key splits for a tensor-core pass with fewer CTAs than SMs
        o1_geom gw = {};
        gw.groups = a.G;
        gw.heads_per_group = a.hpg;
        gw.d = a.d;
        gw.dv = a.dv;
        gw.window = a.w;
        a.wsplit = a.tc ? o1_wsplit(gw, a.R) : 1;
    }
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
    // a short pass takes the short far kernel (stages 1 and 2 stay empty)
    const size_t sfs = short_smem_floats(a) * sizeof(float);
    const bool short_far = R <= O1_SHORT_ROWS && sfs <= 227 * 1024;
    a.far_copy = short_far && a.commit && !a.exact;
    begin(1, sf);
    const size_t fbs = far_block_smem_floats() * sizeof(float);
    if (!a.exact && !short_far) {   // the comparator has no far field
        if (a.dv <= 128) k_far_block<1><<<dim3(nblk, a.nh), 256, fbs, sf>>>(a);   // behind the fork: plain
        else k_far_block<2><<<dim3(nblk, a.nh), 256, fbs, sf>>>(a);
    }
    end(1, sf);
    begin(2, sf);
    const size_t n = (size_t)a.nh * a.m * a.dv;
    if (!a.exact && !short_far) o1_launch_chained(a.chain_early, k_far_tscan, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, sf, a);
    end(2, sf);
    begin(3, sf);
    if (short_far) k_side_short<<<dim3(a.nh, short_col_splits(a)), 256, sfs, sf>>>(a);   // behind the fork: plain
    else if (a.exact) {   // the far branch's first kernel: plain
        if (a.dv <= 128) k_side_readout<1><<<dim3(nblk, a.nh), 256, readout_smem(a), sf>>>(a);
        else k_side_readout<2><<<dim3(nblk, a.nh), 256, readout_smem(a), sf>>>(a);
    } else if (a.dv <= 128) {
        o1_launch_chained(a.chain_early, k_side_readout<1>, dim3(nblk, a.nh), dim3(256), readout_smem(a), sf, a);
    } else {
        o1_launch_chained(a.chain_early, k_side_readout<2>, dim3(nblk, a.nh), dim3(256), readout_smem(a), sf, a);
    }
    end(3, sf);
    cudaEventRecord(aux->join, sf);
    begin(4, st);
    if (a.tc) e = o1_launch_gather_tc(a, st);
    end(4, st);
    begin(5, st);
    if (e == cudaSuccess) {
        if (KS) {
            const int nsl = (a.w + R - 1 + KS - 1) / KS;
            o1_launch_chained(a.chain_early, k_near_small, dim3(nsl, a.G), dim3(256), near_small_smem(a, KS), st, a, KS);
            o1_launch_chained(a.chain_early, k_near_small_merge, dim3(R * a.nh, (a.dv + 63) / 64), dim3(256), 0, st, a, nsl);
        } else if (a.tc) {
            e = o1_launch_near_tc(a, st);
        } else {
            const int RB = 32 / a.hpg;
            const dim3 gn((R + RB - 1) / RB, a.G);
            if (a.dv <= 128) o1_launch_chained(a.chain_early, k_near<1>, gn, dim3(256), near_smem(a), st, a);
            else o1_launch_chained(a.chain_early, k_near<2>, gn, dim3(256), near_smem(a), st, a);
        }
    }
    end(5, st);
    // the far branch is joined even when the window launch failed, so that a
    // capture of `st` stays well formed
    cudaStreamWaitEvent(st, aux->join, 0);
    if (e != cudaSuccess) return e;
    begin(6, st);
    k_merge<<<(unsigned)(((size_t)R * a.nh + 7) / 8), 256, 0, st>>>(a);
    end(6, st);
    begin(7, st);
    const int live = R < a.w ? R : a.w;
    if (a.commit) o1_launch_chained(a.chain_early, k_commit, dim3((live + 3) / 4, a.G), dim3(64), 0, st, a);
    end(7, st);
    return cudaGetLastError();
}

// The state-advancing stages of a pass, without the attention: keys
// rotated, the far insert of every key the rows evict (block partials and
// the scan), the surviving rows into the ring, meta and position. Launched
// on one stream; a.commit must be set and a.tc clear. A short pass is two
// launches: the short far kernel, then the ring push, each rotating the
// pass's keys it reads.
cudaError_t o1_launch_commit_pass(const O1Args &a, cudaStream_t st) {
    chunk_attrs();
    const int R = a.R;
    const int nblk = (R + O1_SUB - 1) / O1_SUB;
    O1Args as = a;
    as.short_no_readout = 1;
    const size_t sfs = short_smem_floats(as) * sizeof(float);
    const bool short_far = R <= O1_SHORT_ROWS && sfs <= 227 * 1024;
    if (short_far) {
        // far inserts, then the ring push scheduled under their end
        as.chain_early = 1;
        as.commit_rotates = 1;
        as.far_copy = !a.exact;
        k_side_short<<<dim3(a.nh, short_col_splits(as)), 256, sfs, st>>>(as);
        const int live = R < a.w ? R : a.w;
        o1_launch_chained(as.chain_early, k_commit_rot, dim3(live, a.G), dim3(128), 0, st, as);
        return cudaGetLastError();
    }
    k_rope<<<R, 128, 0, st>>>(a);
    {
        const size_t fbs = far_block_smem_floats() * sizeof(float);
        if (a.dv <= 128) o1_launch_chained(a.chain_early, k_far_block<1>, dim3(nblk, a.nh), dim3(256), fbs, st, a);
        else o1_launch_chained(a.chain_early, k_far_block<2>, dim3(nblk, a.nh), dim3(256), fbs, st, a);
        const size_t n = (size_t)a.nh * a.m * a.dv;
        o1_launch_chained(a.chain_early, k_far_tscan, dim3((unsigned)((n + 255) / 256)), dim3(256), 0, st, a);
    }
    const int live = R < a.w ? R : a.w;
    o1_launch_chained(a.chain_early, k_commit, dim3((live + 3) / 4, a.G), dim3(64), 0, st, a);
    return cudaGetLastError();
}

// Fresh far field and ring: M = -inf, Z = 0, T = 0, ring zeros.
__global__ void k_init_state(O1Args a) {
    const size_t nM = (size_t)a.nh * a.m;
    const size_t nT = nM * a.dv;
    const size_t nK = (size_t)a.G * a.w * a.d, nV = (size_t)a.G * a.w * a.dv;
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    const size_t nTick = (size_t)a.nh + a.G + 1;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < nT + nK + nV + nM; i += stride) {
        if (i < nM) {
            a.M[i] = -INFINITY;
            a.Z[i] = 0.f;
            a.Zlo[i] = 0.f;
        }
        if (i < nTick) a.tick[i] = 0u;
        if (i < nT) a.T[i] = 0.f;
        else if (i < nT + nK) a.ring_k[i - nT] = 0.f;
        else if (i < nT + nK + nV) a.ring_v[i - nT - nK] = 0.f;
    }
}

cudaError_t o1_launch_init(const O1Args &a, cudaStream_t st) {
    k_init_state<<<304, 256, 0, st>>>(a);
    return cudaGetLastError();
}

// One thread: check that every group can rewind `rows` pushes (dory.rs
// dory_o1_back: a full ring steps head back and farl down, a ring not yet
// full drops its newest entry; a full ring stays full), then apply them all
// and move the position back; otherwise change nothing and raise the flag.
__global__ void k_back(O1Args a, int rows) {
    bool ok = a.hdr->pos >= rows;
    for (int g = 0; g < a.G; ++g) {
        const uint32_t len = a.meta[g * 4 + 0], farl = a.meta[g * 4 + 2], wg = a.meta[g * 4 + 3];
        ok = ok && (len == wg ? farl >= (uint32_t)rows : len >= (uint32_t)rows);
    }
    if (!ok) {
        a.hdr->flags |= (uint32_t)O1_FLAG_BACK_REFUSED;
        return;
    }
    for (int g = 0; g < a.G; ++g) {
        uint32_t *mt = a.meta + g * 4;
        const uint32_t wg = mt[3];
        if (mt[0] == wg) {
            mt[1] = (uint32_t)(((long long)mt[1] + wg - (long long)rows % wg) % wg);
            mt[2] -= (uint32_t)rows;
        } else {
            mt[0] -= (uint32_t)rows;
        }
    }
    a.hdr->pos -= rows;
}

cudaError_t o1_launch_back(const O1Args &a, int rows, cudaStream_t st) {
    k_back<<<1, 1, 0, st>>>(a, rows);
    return cudaGetLastError();
}
