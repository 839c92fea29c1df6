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
//    far blocks (O1_TOK_FS per head, one unless configured otherwise, each
//      over a share of the value columns): the evicted key's far insert
//      fused with the far readout, which reads the updated T once; T is
//      updated in place, and so are M and Z with one block per head (with
//      several, they go through the far record to the merge).
//  k_tok_merge  launched with programmatic dependent launch: waits for the
//      main grid, merges the slices and the far part under one exponent
//      (1e-30 floor), gates, and one block commits ring slot, meta and
//      position.
// Nothing waits on a flag: the only dependency is the launch order.
//
// The step is latency-bound (a few MB, read once): every block issues its
// global loads first, all at once (the row's inputs, bulk copies of the
// large operands), and the dot products run lane-per-key / lane-per-landmark
// over a warp's share of d, so that no reduction waits on a chain of
// shuffles.
#include <math.h>

#include "o1_common.cuh"

__device__ __forceinline__ void o1_allow_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }
__device__ __forceinline__ void o1_wait_primary() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

static size_t tok_near_floats(const O1Args &a) {
    return 4 + (size_t)(a.hpg + 1) * a.d + (size_t)a.KC * (a.d + a.dv) + (size_t)a.KC * a.hpg + 2 * a.hpg +
           (size_t)8 * a.KC * a.hpg;
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
    const size_t m = a.m, cps = o1_tok_far_cols(a.dv);
    return 4 + 2 * (size_t)a.d + a.dv + 2 * m * a.d + m * cps + m * (m + 1) + 16 * m + 4 * m + 4 + 256;
}

static size_t tok_main_smem(const O1Args &a) {
    const size_t n = tok_near_floats(a), f = tok_far_floats(a);
    return 4 * (n > f ? n : f);
}

// Rotary angle of pair j at the row's position (identity when the layer
// does not rotate).
__device__ __forceinline__ void tok_cs(const O1Args &a, float inv, long long p, float &cs, float &sn) {
    cs = 1.f;
    sn = 0.f;
    if (a.rotate) o1_rope_cs(inv, p, cs, sn);
}

// Dot products of `n` rows of shared memory (rows of d floats, `rows`
// apart) with `nq` vectors (d floats, `qstride` apart), lane = row, warp =
// a contiguous share of d in float4 units, visited from a lane-dependent
// start so that the 8 lanes of a quarter warp read 8 different bank groups.
// Returns the warp's partial dots in acc[0 .. nq-1] (0 for lanes >= n).
template <int NQ>
__device__ __forceinline__ void tok_dots(const float *rows, int row, bool valid, const float *qs, int qstride,
                                         int nq, int d, float (&acc)[NQ]) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nu = d >> 2, U = (nu + 7) >> 3;   // U <= 8 for d <= 256
    const int ub = warp * U;
#pragma unroll
    for (int h = 0; h < NQ; ++h) acc[h] = 0.f;
    if (!valid) return;
    const float4 *kr = (const float4 *)(rows + (size_t)row * d);
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    // the row's units first, all in flight, then each vector's
    float4 kv[8];
    int us[8];
    int s = lane % U;
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        us[t] = ub + s;
        kv[t] = (t < U && us[t] < nu) ? kr[us[t]] : z;
        if (++s == U) s = 0;
    }
#pragma unroll
    for (int h = 0; h < NQ; ++h) {
        if (h >= nq) break;
        const float4 *qh = (const float4 *)(qs + (size_t)h * qstride);
        float4 qv[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) qv[t] = (t < U && us[t] < nu) ? qh[us[t]] : z;
        float a0 = 0.f;
#pragma unroll
        for (int t = 0; t < 8; ++t)
            a0 = fmaf(qv[t].x, kv[t].x, fmaf(qv[t].y, kv[t].y, fmaf(qv[t].z, kv[t].z, fmaf(qv[t].w, kv[t].w, a0))));
        acc[h] = a0;
    }
}

__device__ void tok_near(const O1Args &a, int g, int c, const O1Meta &mt, float *sm) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int d = a.d, dv = a.dv, hpg = a.hpg, KC = a.KC;
    const bool evict = mt.len0 == mt.wg;
    const int len1 = evict ? mt.wg : mt.len0 + 1;
    const int head1 = evict ? (mt.head0 + 1) % mt.wg : mt.head0;
    const int n = a.ns + len1;
    const int i0 = c * KC;
    const int cnt = max(0, min(KC, n - i0));
    const size_t slot = (size_t)(g * a.NC + c) * hpg;
    float *pv = a.part + slot * dv;   // [hpg][dv]
    float *pml = a.pml + slot * 2;    // [hpg][2]

    uint64_t *sbar = (uint64_t *)sm;   // the slice's copy barrier
    float *sq = sm + 4;                // [hpg][d]
    float *sk = sq + hpg * d;          // [d]
    float *sK = sk + d;                // [KC][d]
    float *sV = sK + KC * d;           // [KC][dv]
    float *sS = sV + KC * dv;          // [KC][hpg]
    float *sML = sS + KC * hpg;        // [hpg][2]
    float *sP = sML + 2 * hpg;         // [8 warps][KC][hpg] partial dots

    if (cnt == 0 && c != 0) {
        for (int h = tid; h < hpg; h += blockDim.x) {
            pml[2 * h] = -INFINITY;
            pml[2 * h + 1] = 0.f;
        }
        return;
    }
    // the row's inputs first, every load in flight at once: position, the
    // rotary frequency of pair j = tid, the group's queries and key at j and
    // j + d/2, the row's value
    const int half = d >> 1;
    const bool rj = tid < half;
    const long long p = a.hdr->pos;
    const float inv = rj ? a.hdr->inv_freq[tid] : 0.f;
    float x0[O1_MAX_HPG + 1], x1[O1_MAX_HPG + 1];
#pragma unroll
    for (int h = 0; h <= O1_MAX_HPG; ++h) {
        const float *src = h < hpg ? a.q + (size_t)(g * hpg + h) * d : a.k + (size_t)g * d;
        const bool in = rj && h <= hpg;
        x0[h] = in ? src[tid] : 0.f;
        x1[h] = in ? src[tid + half] : 0.f;
    }
    const int ipush = a.ns + len1 - 1 - i0;
    const bool has_push = ipush >= 0 && ipush < cnt;
    float4 vpush = make_float4(0.f, 0.f, 0.f, 0.f);
    if (has_push && tid < (dv >> 2)) vpush = ((const float4 *)(a.v + (size_t)g * dv))[tid];
    // The slice's keys and values: sinks, then ring logical 0..len1-1, as at
    // most three contiguous runs (the sinks, the ring up to its end, the ring
    // from slot 0), each one bulk copy for K and one for V. The last logical
    // key is the pushed one: its slot is overwritten by this row, so its key
    // row is replaced by the row's own rotated key (sk) and its value row by
    // the row's value once the copies have landed.
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
    if (rj) {
        float cs, sn;
        tok_cs(a, inv, p, cs, sn);
#pragma unroll
        for (int h = 0; h <= O1_MAX_HPG; ++h) {
            if (h > hpg) break;
            float *dst = h < hpg ? sq + h * d : sk;
            dst[tid] = x0[h] * cs - x1[h] * sn;
            dst[tid + half] = x1[h] * cs + x0[h] * sn;
        }
    }
    __syncthreads();   // the barrier is initialised before anyone waits on it
    tok_wait_copies(a, sbar);
    if (c == 0)
        for (int j = tid; j < d; j += blockDim.x) a.kcur[(size_t)g * d + j] = sk[j];
    if (has_push) {
        for (int j = tid; j < d; j += blockDim.x) sK[ipush * d + j] = sk[j];
        if (tid < (dv >> 2)) ((float4 *)(sV + (size_t)ipush * dv))[tid] = vpush;   // dv <= 4 * blockDim
    }
    __syncthreads();
    // scores: partial dots per warp (lane = key), then their sum per (key, head)
    for (int k0 = 0; k0 < cnt; k0 += 32) {
        float acc[O1_MAX_HPG];
        const int key = k0 + lane;
        tok_dots(sK, key, key < cnt, sq, d, hpg, d, acc);
        if (key < cnt)
#pragma unroll
            for (int h = 0; h < O1_MAX_HPG; ++h) {
                if (h >= hpg) break;
                sP[((size_t)warp * KC + key) * hpg + h] = acc[h];
            }
    }
    __syncthreads();
    for (int idx = tid; idx < cnt * hpg; idx += blockDim.x) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) s += sP[(size_t)w * KC * hpg + idx];
        sS[idx] = s * a.scale;
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
            pml[2 * h] = mx;
            pml[2 * h + 1] = l;
        }
    }
    __syncthreads();
    // value sums: thread per (head, 4 columns)
    const int dv4 = dv >> 2;
    for (int idx = tid; idx < hpg * dv4; idx += blockDim.x) {
        const int h = idx / dv4, c4 = idx - h * dv4;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int i = 0; i < cnt; ++i) {
            const float w = sS[i * hpg + h];
            const float4 v = ((const float4 *)(sV + (size_t)i * dv))[c4];
            acc.x = fmaf(w, v.x, acc.x);
            acc.y = fmaf(w, v.y, acc.y);
            acc.z = fmaf(w, v.z, acc.z);
            acc.w = fmaf(w, v.w, acc.w);
        }
        ((float4 *)(pv + (size_t)h * dv))[c4] = acc;
    }
}

// Far split fs of head (g, hl): the insert of the evicted key and the
// readout, with the value sums of columns [fs * cps, fs * cps + cps) only.
// Every split computes the landmark part (scores, insert, u, gains, D) in
// full; split 0 records c_f, D and have. With one split per head the block
// writes the new M and Z itself; with several, split 0 puts them in the far
// record and the merge kernel writes them once every block has read the old
// ones.
__device__ void tok_far(const O1Args &a, int g, int hl, int fs, const O1Meta &mt, float *sm) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int d = a.d, dv = a.dv, m = a.m;
    const int h = g * a.hpg + hl;
    const int cps = o1_tok_far_cols(dv), t0 = fs * cps;
    const int ncol = max(0, min(cps, dv - t0));
    const bool evict = mt.len0 == mt.wg;
    const int farl1 = mt.farl0 + (evict ? 1 : 0);
    float *fp = a.farp + (size_t)h * (4 + dv + 2 * m);
    if (farl1 == 0) {   // no far field: an empty record (the merge multiplies the numerator by 0)
        for (int c = tid; c < ncol; c += blockDim.x) fp[4 + t0 + c] = 0.f;
        if (fs == 0 && tid == 0) {
            fp[0] = -INFINITY;
            fp[1] = fp[2] = fp[3] = 0.f;
        }
        return;
    }
    uint64_t *sbar = (uint64_t *)sm;   // the block's copy barrier
    float *sq = sm + 4;                // [d]
    float *ske = sq + d;               // [d]
    float *sve = ske + d;              // [dv]
    float *sqt = sve + dv;             // [m][d]  landmark queries of this head
    float *skt = sqt + m * d;          // [m][d]  landmark keys of the group
    float *sT = skt + m * d;           // [m][cps] this split's value sums
    float *smu = sT + m * cps;         // [m][m + 1]
    float *sP = smu + m * (m + 1);     // [8 warps][m][2] partial dots
    float *se = sP + 16 * m;           // [m] e^{f - F}
    float *sG = se + m;                // [m] gains
    float *sRho = sG + m;              // [m]
    float *sE = sRho + m;              // [m]
    float *sRed = sE + m;              // [4] c_f, D
    float *sNum = sRed + 4;            // [256] numerator partials

    // inputs first: position, frequency and query pair j = tid, the far max
    // and mass (warp 0, landmarks lane and lane + 32), this split's value
    // sums and the mixing matrix by plain loads, the large operands by bulk
    // copies
    const int half = d >> 1;
    const bool rj = tid < half;
    const long long p = a.hdr->pos;
    const float inv = rj ? a.hdr->inv_freq[tid] : 0.f;
    const float qa = rj ? a.q[(size_t)h * d + tid] : 0.f, qb = rj ? a.q[(size_t)h * d + tid + half] : 0.f;
    float Mo[2] = {-INFINITY, -INFINITY}, Zo[2] = {0.f, 0.f};
    if (warp == 0)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int b = lane + 32 * r;
            if (b < m) {
                Mo[r] = a.M[(size_t)h * m + b];
                Zo[r] = a.Z[(size_t)h * m + b];
            }
        }
    if (tid == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(tok_su32(sbar)) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        tok_bulk(sqt, a.qt + (size_t)h * m * d, (uint32_t)m * d * 4, sbar);
        tok_bulk(skt, a.kt + (size_t)g * m * d, (uint32_t)m * d * 4, sbar);
        if (cps == dv) tok_bulk(sT, a.T + (size_t)h * m * dv, (uint32_t)m * dv * 4, sbar);   // all columns: one run
        if (evict) {
            tok_bulk(ske, a.ring_k + ((size_t)g * a.w + mt.head0) * d, (uint32_t)d * 4, sbar);
            tok_bulk(sve, a.ring_v + ((size_t)g * a.w + mt.head0) * dv, (uint32_t)dv * 4, sbar);
        }
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tok_su32(sbar)) : "memory");
    }
    // a share of T's columns and the mixing matrix by plain loads, every
    // load issued before any store
    if (cps != dv)
        for (int i0 = 0; i0 < m * cps; i0 += 8 * blockDim.x) {
            float tv[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int idx = i0 + u * blockDim.x + tid, b = idx / cps, c = idx - b * cps;
                tv[u] = (idx < m * cps && c < ncol) ? a.T[((size_t)h * m + b) * dv + t0 + c] : 0.f;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u)
                if (i0 + u * blockDim.x + tid < m * cps) sT[i0 + u * blockDim.x + tid] = tv[u];
        }
    for (int i0 = 0; i0 < m * m; i0 += 8 * blockDim.x) {
        float mv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int idx = i0 + u * blockDim.x + tid;
            mv[u] = idx < m * m ? a.mu[(size_t)h * m * m + idx] : 0.f;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int idx = i0 + u * blockDim.x + tid, aa = idx / m;
            if (idx < m * m) smu[aa * (m + 1) + (idx - aa * m)] = mv[u];
        }
    }
    if (rj) {
        float cs, sn;
        tok_cs(a, inv, p, cs, sn);
        sq[tid] = qa * cs - qb * sn;
        sq[tid + half] = qb * cs + qa * sn;
    }
    __syncthreads();   // the barrier is initialised before anyone waits on it
    tok_wait_copies(a, sbar);
    if (!evict)
        for (int j = tid; j < d; j += blockDim.x) ske[j] = 0.f;   // no insert: its logits are unused
    __syncthreads();
    // partial dots per warp, lane = landmark: qt_b . k_e (the insert) and
    // kt_b . q' (the readout)
    for (int b0 = 0; b0 < m; b0 += 32) {
        const int b = b0 + lane;
        float s1[1], s2[1];
        tok_dots(sqt, b, b < m, ske, 0, 1, d, s1);
        tok_dots(skt, b, b < m, sq, 0, 1, d, s2);
        if (b < m) {
            sP[((size_t)warp * m + b) * 2] = s1[0];
            sP[((size_t)warp * m + b) * 2 + 1] = s2[0];
        }
    }
    __syncthreads();
    // warp 0, landmarks lane and lane + 32: the insert of the evicted key
    // (o1b_far_e / o1b_far_commit for one row), the readout's u, gains and D
    if (warp == 0) {
        float f[2], Mn[2], Zn[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int b = lane + 32 * r;
            f[r] = -INFINITY;
            Mn[r] = -INFINITY;
            Zn[r] = 0.f;
            if (b < m) {
                float s = 0.f, ff = 0.f;
#pragma unroll
                for (int w = 0; w < 8; ++w) {
                    s += sP[((size_t)w * m + b) * 2];
                    ff += sP[((size_t)w * m + b) * 2 + 1];
                }
                f[r] = ff * a.scale;
                float rho = 1.f, e = 0.f;
                Mn[r] = Mo[r];
                Zn[r] = Zo[r];
                if (evict) {
                    const float l = s * a.scale;
                    Mn[r] = fmaxf(Mo[r], l);
                    rho = (Mn[r] == Mo[r]) ? 1.f : expf(Mo[r] - Mn[r]);
                    e = expf(l - Mn[r]);
                    Zn[r] = Zo[r] * rho + e;
                    if (O1_TOK_FS == 1) {
                        // the only block of this head that reads M and Z
                        a.M[(size_t)h * m + b] = Mn[r];
                        a.Z[(size_t)h * m + b] = Zn[r];
                    } else if (fs == 0) {
                        fp[4 + dv + b] = Mn[r];
                        fp[4 + dv + m + b] = Zn[r];
                    }
                }
                sRho[b] = rho;
                sE[b] = e;
            }
        }
        const float F = warp_max(fmaxf(f[0], f[1]));
#pragma unroll
        for (int r = 0; r < 2; ++r)
            if (lane + 32 * r < m) se[lane + 32 * r] = expf(f[r] - F);
        __syncwarp();
        float u[2] = {0.f, 0.f}, cb[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int b = lane + 32 * r;
            if (b < m) {
                float acc = 0.f;
                for (int aa = 0; aa < m; ++aa) acc = fmaf(se[aa], smu[aa * (m + 1) + b], acc);
                u[r] = a.rect ? fmaxf(acc, 0.f) : acc;
                cb[r] = F + Mn[r];
            }
        }
        const float cf = warp_max(fmaxf(cb[0], cb[1]));
        float D = 0.f;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int b = lane + 32 * r;
            if (b < m) {
                const float gn = u[r] * expf(cb[r] - cf);
                sG[b] = gn;
                D = fmaf(gn, Zn[r], D);
            }
        }
        D = warp_sum(D);
        if (lane == 0) {
            sRed[0] = cf;
            sRed[1] = D;
        }
    }
    __syncthreads();
    const float cf = sRed[0], D = sRed[1];
    const bool have = D >= 0.f;
    // this split's value sums: thread = (column c, landmark group lg); insert
    // the evicted value, write T back, partial far numerators, then their sum
    const int nlg = blockDim.x / cps, c = tid % cps, lg = tid / cps;
    if (lg < nlg) {
        const float vt = (evict && c < ncol) ? sve[t0 + c] : 0.f;
        float acc = 0.f;
        for (int b = lg; b < m; b += nlg) {
            float x = sT[b * cps + c];
            if (evict) {
                x = sRho[b] * x + sE[b] * vt;
                if (c < ncol) a.T[((size_t)h * m + b) * dv + t0 + c] = x;
            }
            acc = fmaf(sG[b], x, acc);
        }
        sNum[lg * cps + c] = acc;
    }
    __syncthreads();
    if (tid < ncol) {
        float acc = 0.f;
        for (int q = 0; q < nlg; ++q) acc += sNum[q * cps + tid];
        fp[4 + t0 + tid] = have ? acc : 0.f;
    }
    if (fs == 0 && tid == 0) {
        fp[0] = cf;
        fp[1] = have ? D : 0.f;
        fp[2] = have ? 1.f : 0.f;
        fp[3] = evict ? 1.f : 0.f;
    }
}

__global__ __launch_bounds__(256) void k_tok_main(O1Args a) {
    extern __shared__ __align__(16) float sm[];
    o1_allow_dependents();
    const int per = a.NC + a.hpg * O1_TOK_FS;
    const int g = blockIdx.x / per, r = blockIdx.x % per;
    const O1Meta mt = o1_meta(a, g);
    if (r < a.NC) tok_near(a, g, r, mt, sm);
    else tok_far(a, g, (r - a.NC) / O1_TOK_FS, (r - a.NC) % O1_TOK_FS, mt, sm);
}

// Merge per (head, 32 value columns), 256 threads = 8 slice groups x 32
// columns, in one pass over the slices with an online max, 16 slices' loads
// per thread in flight at once (each group keeps its own max, sum and value
// sum, combined at the end); block (0, 0) also commits the row.
__global__ __launch_bounds__(256) void k_tok_merge(O1Args a) {
    __shared__ float smx[8][32], sl[8][32], sacc[8][32];
    const int tid = threadIdx.x;
    const int h = blockIdx.x, g = h / a.hpg, hl = h % a.hpg;
    const int sgp = tid >> 5, col = tid & 31, t = blockIdx.y * 32 + col;
    const size_t base = (size_t)g * a.NC * a.hpg + hl;   // (slice c) -> base + c * hpg
    // the gate is this call's input, not the main grid's output: read it
    // before waiting
    const float gl = (sgp == 0 && a.gate && t < a.dv) ? a.gate[(size_t)h * a.dv + t] : 0.f;
    o1_wait_primary();
    const size_t fstride = 4 + (size_t)a.dv + 2 * (size_t)a.m;
    const float *fp = a.farp + (size_t)h * fstride;
    float cf = -INFINITY, Df = 0.f, hv = 0.f, fnum = 0.f;
    if (sgp == 0) {   // the far part, in the same round as the slices' partials
        cf = __ldcg(fp);
        Df = __ldcg(fp + 1);
        hv = __ldcg(fp + 2);
        fnum = t < a.dv ? __ldcg(fp + 4 + t) : 0.f;
    }
    float mx = -INFINITY, l = 0.f, acc = 0.f;
    for (int c0 = sgp; c0 < a.NC; c0 += 8 * 16) {
        float mc[16], lc[16], vc[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            const int c = c0 + 8 * u;
            const bool in = c < a.NC;
            const size_t sl_ = base + (size_t)c * a.hpg;
            mc[u] = in ? __ldcg(a.pml + 2 * sl_) : -INFINITY;
            lc[u] = in ? __ldcg(a.pml + 2 * sl_ + 1) : 0.f;
            vc[u] = (in && t < a.dv) ? __ldcg(a.part + sl_ * a.dv + t) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < 16; ++u) {
            if (mc[u] == -INFINITY) continue;
            const float mn = fmaxf(mx, mc[u]);
            const float fo = expf(mx - mn), fc = expf(mc[u] - mn);
            l = l * fo + lc[u] * fc;
            acc = acc * fo + vc[u] * fc;
            mx = mn;
        }
    }
    smx[sgp][col] = mx;
    sl[sgp][col] = l;
    sacc[sgp][col] = acc;
    __syncthreads();
    if (sgp == 0 && t < a.dv) {
        float M = -INFINITY;
#pragma unroll
        for (int q = 0; q < 8; ++q) M = fmaxf(M, smx[q][col]);
        float L = 0.f, A = 0.f;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            if (smx[q][col] == -INFINITY) continue;
            const float f = expf(smx[q][col] - M);
            L = fmaf(sl[q][col], f, L);
            A = fmaf(sacc[q][col], f, A);
        }
        const bool have = hv > 0.5f;
        const float c = cf > -INFINITY ? fmaxf(M, cf) : M;
        const float al = expf(M - c);
        const float be = have ? expf(cf - c) : 0.f;
        const float den = fmaxf(be * Df + al * L, 1e-30f);
        float y = (be * fnum + al * A) / den;
        if (a.gate) y = y / (1.f + expf(-gl));
        a.out[(size_t)h * a.dv + t] = y;
    }
    if (O1_TOK_FS > 1 && blockIdx.y == 0 && __ldcg(fp + 3) > 0.5f) {
        // the far insert's new max and mass (written by far split 0), now
        // that every block of the main grid has read the old ones
        for (int b = tid; b < a.m; b += blockDim.x) {
            a.M[(size_t)h * a.m + b] = __ldcg(fp + 4 + a.dv + b);
            a.Z[(size_t)h * a.m + b] = __ldcg(fp + 4 + a.dv + a.m + b);
        }
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
    static unsigned long long done = 0;
    unsigned long long bit = 0;
    if (o1_attrs_needed(&done, &bit)) {
        cudaFuncSetAttribute(k_tok_main, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        o1_attrs_done(&done, bit);
    }
    k_tok_main<<<a.G * (a.NC + a.hpg * O1_TOK_FS), 256, tok_main_smem(a), st>>>(a);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.nh, (a.dv + 31) / 32, 1);
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
