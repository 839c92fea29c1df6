// The one-row (decode) path of a sealed O(1) layer: rope, far insert, ring
// push, attend, gate for a single row, in two launches.
//
// The pages' one-row path ("cortiq-engine 0.8.82 src/gpu_metal/o1c.rs",
// encode_tok: near partials split over threadgroups, the far part per query
// head, a merge, a commit; "cortiq-engine 0.8.77 src/gpu_wgpu/dory.rs",
// dory_os ... dory_ogate with the engine's far insert and push before them)
// is four to nine dispatches. Here:
//
//  k_tok_main   blockIdx -> (group, role):
//    near blocks: KC keys of the group's near set after the push (sinks,
//      then ring logical 0..len'-1; the pushed slot is served from the
//      row's own rotated key and value, so the ring is not written before
//      every block has read it), scores for every head of the group, a
//      slice-local softmax -> partial (max, sum, value sum) per head.
//    far blocks (one per head): the evicted key's far insert (M, Z, T in
//      place) fused with the far readout, which reads the updated T once.
//  k_tok_merge  launched with programmatic dependent launch: waits for the
//      main grid, merges the slices and the far part under one exponent
//      (1e-30 floor), gates, and one block commits ring slot, meta and
//      position.
// Nothing waits on a flag: the only dependency is the launch order.
//
// The step is latency-bound (a few MB, read once), so every block issues its
// global loads in one batch (many in flight, no integer division in the
// address arithmetic) before computing from shared memory.
#include <math.h>

#include "o1_common.cuh"

__device__ __forceinline__ void o1_allow_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }
__device__ __forceinline__ void o1_wait_primary() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

static size_t tok_near_floats(const O1Args &a) {
    return 4 + (size_t)(a.hpg + 1) * a.d + (size_t)a.KC * (a.d + a.dv) + (size_t)a.KC * a.hpg + 2 * a.hpg;
}

// Bulk copies into shared memory completing on one mbarrier: thread 0 adds
// each copy's bytes and issues it; everyone waits (bounded, about 2 s).
__device__ __forceinline__ uint32_t tok_su32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void tok_bulk(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    if (!bytes) return;
    asm volatile("mbarrier.expect_tx.shared::cta.b64 [%0], %1;" ::"r"(tok_su32(bar)), "r"(bytes) : "memory");
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     tok_su32(dst)),
                 "l"((uint64_t)src), "r"(bytes), "r"(tok_su32(bar))
                 : "memory");
}
__device__ __forceinline__ bool tok_wait(uint64_t *bar) {
    const long long t0 = clock64();
    while (true) {
        uint32_t ok;
        asm volatile(
            "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\nselp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(ok)
            : "r"(tok_su32(bar))
            : "memory");
        if (ok) return true;
        if (clock64() - t0 > 4000000000LL) return false;
    }
}
// Waits for the block's copies; on expiry raises the flag and waits once more
// for the copies still in flight (they write this block's shared memory).
__device__ __forceinline__ void tok_wait_copies(const O1Args &a, uint64_t *bar) {
    if (!tok_wait(bar)) {
        if (threadIdx.x == 0) atomicOr(&a.hdr->flags, (uint32_t)O1_FLAG_WAIT_EXPIRED);
        tok_wait(bar);
    }
}

static size_t tok_far_floats(const O1Args &a) {
    const size_t m = a.m;
    return 4 + 2 * (size_t)a.d + a.dv + 2 * m * a.d + m * (m + 1) + m * a.dv + 11 * m + 32;
}

static size_t tok_main_smem(const O1Args &a) {
    const size_t n = tok_near_floats(a), f = tok_far_floats(a);
    return 4 * (n > f ? n : f);
}

// Rotates the rows xs[0 .. n-1] (global, d wide) into dst[r] (shared) at
// position p: pair (j, j + d/2), one angle per j for all rows.
__device__ __forceinline__ void tok_rotate(const O1Args &a, long long p, const float *const *xs, float *const *dst,
                                           int n) {
    const int half = a.d >> 1;
    for (int j = threadIdx.x; j < half; j += blockDim.x) {
        float cs = 1.f, sn = 0.f;
        if (a.rotate) o1_rope_cs(a.hdr->inv_freq[j], p, cs, sn);
        for (int h0 = 0; h0 < n; h0 += 8) {
            float x0[8], x1[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const bool in = h0 + u < n;
                x0[u] = in ? xs[h0 + u][j] : 0.f;
                x1[u] = in ? xs[h0 + u][j + half] : 0.f;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (h0 + u >= n) break;
                dst[h0 + u][j] = x0[u] * cs - x1[u] * sn;
                dst[h0 + u][j + half] = x1[u] * cs + x0[u] * sn;
            }
        }
    }
}

__device__ void tok_near(const O1Args &a, int g, int c, const O1Meta &mt, float *sm) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int d = a.d, dv = a.dv, hpg = a.hpg;
    const bool evict = mt.len0 == mt.wg;
    const int len1 = evict ? mt.wg : mt.len0 + 1;
    const int head1 = evict ? (mt.head0 + 1) % mt.wg : mt.head0;
    const int n = a.ns + len1;
    const int i0 = c * a.KC;
    const int cnt = max(0, min(a.KC, n - i0));
    float *part = a.part + (size_t)(g * a.NC + c) * hpg * (2 + dv);

    uint64_t *sbar = (uint64_t *)sm;   // the slice's copy barrier
    float *sq = sm + 4;                // [hpg][d]
    float *sk = sq + hpg * d;          // [d]
    float *sK = sk + d;                // [KC][d]
    float *sV = sK + a.KC * d;         // [KC][dv]
    float *sS = sV + a.KC * dv;        // [KC][hpg]
    float *sML = sS + a.KC * hpg;      // [hpg][2]

    if (cnt == 0 && c != 0) {
        for (int idx = tid; idx < hpg * (2 + dv); idx += blockDim.x) {
            const int e = idx % (2 + dv);
            part[idx] = e == 0 ? -INFINITY : 0.f;
        }
        return;
    }
    // The slice's keys and values: sinks, then ring logical 0..len1-1, as at
    // most three contiguous runs (the sinks, the ring up to its end, the ring
    // from slot 0), each one bulk copy for K and one for V. The last logical
    // key is the pushed one: its slot is overwritten by this row, so its key
    // row is replaced by the row's own rotated key (sk) and its value row by
    // the row's value once the copies have landed.
    const int ipush = a.ns + len1 - 1 - i0;
    if (tid == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(tok_su32(sbar)) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        const int nsk = max(0, min(cnt, a.ns - i0));   // sink entries of the slice
        if (nsk > 0) {
            tok_bulk(sK, a.sink_k + ((size_t)g * a.ns + i0) * d, (uint32_t)nsk * d * 4, sbar);
            tok_bulk(sV, a.sink_v + ((size_t)g * a.ns + i0) * dv, (uint32_t)nsk * dv * 4, sbar);
        }
        const int nr = cnt - nsk;                      // ring entries of the slice
        if (nr > 0) {
            const int L0 = i0 + nsk - a.ns;            // first logical ring index
            const int s0 = (head1 + L0) % mt.wg;
            const int na = min(nr, mt.wg - s0);
            tok_bulk(sK + (size_t)nsk * d, a.ring_k + ((size_t)g * a.w + s0) * d, (uint32_t)na * d * 4, sbar);
            tok_bulk(sV + (size_t)nsk * dv, a.ring_v + ((size_t)g * a.w + s0) * dv, (uint32_t)na * dv * 4, sbar);
            if (nr > na) {
                tok_bulk(sK + (size_t)(nsk + na) * d, a.ring_k + (size_t)g * a.w * d, (uint32_t)(nr - na) * d * 4, sbar);
                tok_bulk(sV + (size_t)(nsk + na) * dv, a.ring_v + (size_t)g * a.w * dv, (uint32_t)(nr - na) * dv * 4,
                         sbar);
            }
        }
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tok_su32(sbar)) : "memory");
    }
    // rotate the group's queries and its key while the copies are in flight
    {
        const float *xs[O1_MAX_HPG + 1];
        float *dst[O1_MAX_HPG + 1];
        for (int h = 0; h < hpg; ++h) {
            xs[h] = a.q + (size_t)(g * hpg + h) * d;
            dst[h] = sq + h * d;
        }
        xs[hpg] = a.k + (size_t)g * d;
        dst[hpg] = sk;
        tok_rotate(a, a.hdr->pos, xs, dst, hpg + 1);
    }
    float4 vpush = make_float4(0.f, 0.f, 0.f, 0.f);
    const bool has_push = ipush >= 0 && ipush < cnt;
    if (has_push && tid < (dv >> 2)) vpush = ((const float4 *)(a.v + (size_t)g * dv))[tid];
    __syncthreads();   // the barrier is initialised before anyone waits on it
    tok_wait_copies(a, sbar);
    if (c == 0)
        for (int j = tid; j < d; j += blockDim.x) a.kcur[(size_t)g * d + j] = sk[j];
    if (has_push) {
        for (int j = tid; j < d; j += blockDim.x) sK[ipush * d + j] = sk[j];
        if (tid < (dv >> 2)) ((float4 *)(sV + (size_t)ipush * dv))[tid] = vpush;   // dv <= 4 * blockDim
    }
    if (cnt == 0) return;   // slice 0 of an empty set only publishes the key
    __syncthreads();
    // scores: one warp per key, lanes across d (dense rows, conflict-free),
    // every head of the group at once
    for (int i = warp; i < cnt; i += blockDim.x >> 5) {
        float acc[O1_MAX_HPG];
#pragma unroll
        for (int h = 0; h < O1_MAX_HPG; ++h) acc[h] = 0.f;
        for (int j4 = lane; j4 < (d >> 2); j4 += 32) {
            const float4 kv = ((const float4 *)(sK + (size_t)i * d))[j4];
#pragma unroll
            for (int h = 0; h < O1_MAX_HPG; ++h) {
                if (h >= hpg) break;
                const float4 qv = ((const float4 *)(sq + h * d))[j4];
                acc[h] = fmaf(qv.x, kv.x, fmaf(qv.y, kv.y, fmaf(qv.z, kv.z, fmaf(qv.w, kv.w, acc[h]))));
            }
        }
#pragma unroll
        for (int h = 0; h < O1_MAX_HPG; ++h) {
            if (h >= hpg) break;
            const float sh = warp_sum(acc[h]);
            if (lane == 0) sS[i * hpg + h] = sh * a.scale;
        }
    }
    __syncthreads();
    // slice-local softmax per head
    for (int h = warp; h < hpg; h += blockDim.x >> 5) {
        float mx = -INFINITY;
        for (int i = lane; i < cnt; i += 32) mx = fmaxf(mx, sS[i * hpg + h]);
        mx = warp_max(mx);
        float l = 0.f;
        for (int i = lane; i < cnt; i += 32) {
            const float e = expf(sS[i * hpg + h] - mx);
            sS[i * hpg + h] = e;
            l += e;
        }
        l = warp_sum(l);
        if (lane == 0) {
            sML[2 * h] = mx;
            sML[2 * h + 1] = l;
        }
    }
    __syncthreads();
    // value sums: thread per (head, column), two accumulators
    for (int idx = tid; idx < hpg * dv; idx += blockDim.x) {
        const int h = idx / dv, t = idx - h * dv;
        float acc0 = 0.f, acc1 = 0.f;
        int i = 0;
        for (; i + 1 < cnt; i += 2) {
            acc0 = fmaf(sS[i * hpg + h], sV[i * dv + t], acc0);
            acc1 = fmaf(sS[(i + 1) * hpg + h], sV[(i + 1) * dv + t], acc1);
        }
        if (i < cnt) acc0 = fmaf(sS[i * hpg + h], sV[i * dv + t], acc0);
        part[h * (2 + dv) + 2 + t] = acc0 + acc1;
    }
    for (int h = tid; h < hpg; h += blockDim.x) {
        part[h * (2 + dv)] = sML[2 * h];
        part[h * (2 + dv) + 1] = sML[2 * h + 1];
    }
}

__device__ void tok_far(const O1Args &a, int g, int hl, const O1Meta &mt, float *sm) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
    const int d = a.d, dv = a.dv, m = a.m;
    const int h = g * a.hpg + hl;
    const bool evict = mt.len0 == mt.wg;
    const int farl1 = mt.farl0 + (evict ? 1 : 0);
    float *fp = a.farp + (size_t)h * (4 + dv);
    if (farl1 == 0) {
        for (int idx = tid; idx < 4 + dv; idx += blockDim.x) fp[idx] = idx == 0 ? -INFINITY : 0.f;
        return;
    }
    uint64_t *sbar = (uint64_t *)sm;   // the block's copy barrier
    float *sq = sm + 4;            // [d]
    float *ske = sq + d;           // [d]
    float *sve = ske + d;          // [dv]
    float *sqt = sve + dv;         // [m][d]  landmark queries of this head
    float *skt = sqt + m * d;      // [m][d]  landmark keys of the group
    float *sT = skt + m * d;       // [m][dv] value sums
    float *smu = sT + m * dv;      // [m][m + 1]
    float *sMo = smu + m * (m + 1); // [m] far max before the insert
    float *sZo = sMo + m;          // [m]
    float *sMn = sZo + m;          // [m] far max after the insert
    float *sZn = sMn + m;          // [m] far mass after the insert
    float *sRho = sZn + m;         // [m]
    float *sE = sRho + m;          // [m]
    float *sF = sE + m;            // [m] landmark scores, then e^{f - F}
    float *sG = sF + m;            // [m] u, then gains
    float *sC = sG + m;            // [m] F + M_b
    float *sRed = sC + m;          // [32]

    // every large input of the block by bulk copies, the small ones by loads
    if (tid == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(tok_su32(sbar)) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        tok_bulk(sqt, a.qt + (size_t)h * m * d, (uint32_t)m * d * 4, sbar);
        tok_bulk(skt, a.kt + (size_t)g * m * d, (uint32_t)m * d * 4, sbar);
        tok_bulk(sT, a.T + (size_t)h * m * dv, (uint32_t)m * dv * 4, sbar);
        if (evict) {
            tok_bulk(ske, a.ring_k + ((size_t)g * a.w + mt.head0) * d, (uint32_t)d * 4, sbar);
            tok_bulk(sve, a.ring_v + ((size_t)g * a.w + mt.head0) * dv, (uint32_t)dv * 4, sbar);
        }
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tok_su32(sbar)) : "memory");
    }
    for (int i = tid; i < m * m; i += blockDim.x) {
        const int aa = i / m, b = i - aa * m;
        smu[aa * (m + 1) + b] = a.mu[(size_t)h * m * m + i];
    }
    for (int b = tid; b < m; b += blockDim.x) {
        sMo[b] = a.M[(size_t)h * m + b];
        sZo[b] = a.Z[(size_t)h * m + b];
    }
    {
        const float *xs[1] = {a.q + (size_t)h * d};
        float *dst[1] = {sq};
        tok_rotate(a, a.hdr->pos, xs, dst, 1);
    }
    __syncthreads();   // the barrier is initialised before anyone waits on it
    tok_wait_copies(a, sbar);
    // far insert of the evicted key (o1b_far_e / o1b_far_commit for one row)
    // and the landmark scores, one warp per landmark
    for (int b = warp; b < m; b += nw) {
        float s = 0.f;
        if (evict) {
            for (int j = lane; j < d; j += 32) s = fmaf(sqt[b * d + j], ske[j], s);
            s = warp_sum(s);
        }
        float f = 0.f;
        for (int j = lane; j < d; j += 32) f = fmaf(sq[j], skt[b * d + j], f);
        f = warp_sum(f);
        if (lane == 0) {
            const float Mo = sMo[b], Zo = sZo[b];
            if (evict) {
                const float l = s * a.scale;
                const float Mn = fmaxf(Mo, l);
                const float rho = (Mn == Mo) ? 1.f : expf(Mo - Mn);
                const float e = expf(l - Mn);
                sMn[b] = Mn;
                sZn[b] = Zo * rho + e;
                sRho[b] = rho;
                sE[b] = e;
            } else {
                sMn[b] = Mo;
                sZn[b] = Zo;
                sRho[b] = 1.f;
                sE[b] = 0.f;
            }
            sF[b] = f * a.scale;
        }
    }
    __syncthreads();
    if (evict)
        for (int b = tid; b < m; b += blockDim.x) {
            a.M[(size_t)h * m + b] = sMn[b];
            a.Z[(size_t)h * m + b] = sZn[b];
        }
    if (warp == 0) {
        float mx = -INFINITY;
        for (int aa = lane; aa < m; aa += 32) mx = fmaxf(mx, sF[aa]);
        mx = warp_max(mx);
        if (lane == 0) sRed[0] = mx;
    }
    __syncthreads();
    const float F = sRed[0];
    for (int aa = tid; aa < m; aa += blockDim.x) sF[aa] = expf(sF[aa] - F);
    __syncthreads();
    for (int b = tid; b < m; b += blockDim.x) {
        float u = 0.f;
        for (int aa = 0; aa < m; ++aa) u = fmaf(sF[aa], smu[aa * (m + 1) + b], u);
        if (a.rect) u = fmaxf(u, 0.f);
        sG[b] = u;
        sC[b] = F + sMn[b];
    }
    __syncthreads();
    if (warp == 0) {
        float mx = -INFINITY;
        for (int b = lane; b < m; b += 32) mx = fmaxf(mx, sC[b]);
        mx = warp_max(mx);
        float D = 0.f;
        for (int b = lane; b < m; b += 32) {
            const float gn = sG[b] * expf(sC[b] - mx);
            sG[b] = gn;
            D = fmaf(gn, sZn[b], D);
        }
        D = warp_sum(D);
        if (lane == 0) {
            sRed[1] = mx;
            sRed[2] = D;
        }
    }
    __syncthreads();
    const float cf = sRed[1], D = sRed[2];
    const bool have = D >= 0.f;
    // value sums: insert the evicted value, write T back, read the far numerator
    for (int t = tid; t < dv; t += blockDim.x) {
        const float vt = evict ? sve[t] : 0.f;
        float acc = 0.f;
        for (int b = 0; b < m; ++b) {
            float x = sT[b * dv + t];
            if (evict) {
                x = sRho[b] * x + sE[b] * vt;
                a.T[((size_t)h * m + b) * dv + t] = x;
            }
            acc = fmaf(sG[b], x, acc);
        }
        fp[4 + t] = have ? acc : 0.f;
    }
    if (tid == 0) {
        fp[0] = cf;
        fp[1] = have ? D : 0.f;
        fp[2] = have ? 1.f : 0.f;
        fp[3] = 0.f;
    }
}

__global__ __launch_bounds__(256) void k_tok_main(O1Args a) {
    extern __shared__ __align__(16) float sm[];
    o1_allow_dependents();
    const int per = a.NC + a.hpg;
    const int g = blockIdx.x / per, r = blockIdx.x % per;
    const O1Meta mt = o1_meta(a, g);
    if (r < a.NC) tok_near(a, g, r, mt, sm);
    else tok_far(a, g, r - a.NC, mt, sm);
}

// Merge per (head, 64 value columns), 256 threads = 4 slice groups x 64
// columns, in one pass over the slices with an online max (each group keeps
// its own max, sum and value sum, combined at the end); block (0, 0) also
// commits the row.
__global__ __launch_bounds__(256) void k_tok_merge(O1Args a) {
    __shared__ float smx[4][64], sl[4][64], sacc[4][64];
    o1_wait_primary();
    const int tid = threadIdx.x;
    const int h = blockIdx.x, g = h / a.hpg, hl = h % a.hpg;
    const int cg = tid >> 6, col = tid & 63, t = blockIdx.y * 64 + col;
    const size_t cs = (size_t)a.hpg * (2 + a.dv);
    const float *part = a.part + (size_t)g * a.NC * cs + (size_t)hl * (2 + a.dv);
    float mx = -INFINITY, l = 0.f, acc = 0.f;
    for (int c0 = cg; c0 < a.NC; c0 += 16) {
        float mc[4], lc[4], vc[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int c = c0 + 4 * u;
            const bool in = c < a.NC;
            mc[u] = in ? __ldcg(part + c * cs) : -INFINITY;
            lc[u] = in ? __ldcg(part + c * cs + 1) : 0.f;
            vc[u] = (in && t < a.dv) ? __ldcg(part + c * cs + 2 + t) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (mc[u] == -INFINITY) continue;
            const float mn = fmaxf(mx, mc[u]);
            const float fo = expf(mx - mn), fc = expf(mc[u] - mn);
            l = l * fo + lc[u] * fc;
            acc = acc * fo + vc[u] * fc;
            mx = mn;
        }
    }
    smx[cg][col] = mx;
    sl[cg][col] = l;
    sacc[cg][col] = acc;
    __syncthreads();
    if (cg == 0 && t < a.dv) {
        const float M = fmaxf(fmaxf(smx[0][col], smx[1][col]), fmaxf(smx[2][col], smx[3][col]));
        float L = 0.f, A = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            if (smx[q][col] == -INFINITY) continue;
            const float f = expf(smx[q][col] - M);
            L = fmaf(sl[q][col], f, L);
            A = fmaf(sacc[q][col], f, A);
        }
        const float *fp = a.farp + (size_t)h * (4 + a.dv);
        const float cf = __ldcg(fp), Df = __ldcg(fp + 1);
        const bool have = __ldcg(fp + 2) > 0.5f;
        const float c = cf > -INFINITY ? fmaxf(M, cf) : M;
        const float al = expf(M - c);
        const float be = have ? expf(cf - c) : 0.f;
        const float den = fmaxf(be * Df + al * L, 1e-30f);
        float y = (be * __ldcg(fp + 4 + t) + al * A) / den;
        if (a.gate) y = y / (1.f + expf(-a.gate[(size_t)h * a.dv + t]));
        a.out[(size_t)h * a.dv + t] = y;
    }
    if (blockIdx.x == 0 && blockIdx.y == 0) {
        // ring push and meta for every group (o1b_ring_commit / o1b_meta, one row)
        for (int gg = 0; gg < a.G; ++gg) {
            const uint32_t len0 = a.meta[gg * 4 + 0], head0 = a.meta[gg * 4 + 1], wg = a.meta[gg * 4 + 3];
            const uint32_t slot = (head0 + len0) % wg;
            for (int j = threadIdx.x; j < a.d; j += blockDim.x)
                a.ring_k[((size_t)gg * a.w + slot) * a.d + j] = __ldcg(a.kcur + (size_t)gg * a.d + j);
            for (int j = threadIdx.x; j < a.dv; j += blockDim.x)
                a.ring_v[((size_t)gg * a.w + slot) * a.dv + j] = a.v[(size_t)gg * a.dv + j];
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            for (int gg = 0; gg < a.G; ++gg) {
                const uint32_t len0 = a.meta[gg * 4 + 0], head0 = a.meta[gg * 4 + 1], wg = a.meta[gg * 4 + 3];
                if (len0 == wg) {
                    a.meta[gg * 4 + 1] = (head0 + 1) % wg;
                    a.meta[gg * 4 + 2] += 1;
                } else {
                    a.meta[gg * 4 + 0] = len0 + 1;
                }
            }
            a.hdr->pos += 1;
        }
    }
}

cudaError_t o1_launch_token(const O1Args &a, cudaStream_t st) {
    static bool attrs_set = false;
    if (!attrs_set) {
        cudaFuncSetAttribute(k_tok_main, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        attrs_set = true;
    }
    k_tok_main<<<a.G * (a.NC + a.hpg), 256, tok_main_smem(a), st>>>(a);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.nh, (a.dv + 63) / 64, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaLaunchKernelEx(&cfg, k_tok_merge, a);
    return cudaPeekAtLastError();
}
