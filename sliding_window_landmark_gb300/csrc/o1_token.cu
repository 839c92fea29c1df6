// The one-row (decode) path of a sealed O(1) layer: rope, far insert, ring
// push, attend and gate for a single row, in one launch.
//
// The pages' one-row path ("cortiq-engine 0.8.82 src/gpu_metal/o1c.rs",
// encode_tok: near partials split over threadgroups, the far part per query
// head, a merge, a commit; "cortiq-engine 0.8.77 src/gpu_wgpu/dory.rs",
// dory_os ... dory_ogate with the engine's far insert and push before them)
// is four to nine dispatches. Here one grid does all of it:
//
//   far chunks   one CTA per (head, MB landmark queries b): the evicted key's
//                far insert for those b (M, Z, T updated in place; no other
//                CTA of the step reads them) fused with the readout's share:
//                the landmark scores f over every landmark key, u_b, gains,
//                and the chunk's far mass and numerator under its own
//                exponent.
//   near slices  one CTA per (group, KC keys of the near set after the push:
//                sinks, then ring logical 0 .. len' - 1, the pushed slot
//                served from the row's own rotated key and value, so that the
//                ring is not written before every CTA has read it): scores
//                for every head of the group, a slice-local softmax, partial
//                (max, sum, value sum) per head.
//   merge        the last CTA to finish for a head (an arrival counter per
//                head in the state; nothing waits on it) combines that head's
//                slices and far chunks under one exponent, with the 1e-30
//                floor, and gates.
//   commit       the last CTA of a group writes the group's ring slot and
//                meta; the last group moves the position, the step's last
//                write.
//
// Overlap with the previous kernel. The CTAs start while the previous kernel
// on the stream is finishing (programmatic dependent launch) and issue the
// copies of this layer's state before they wait for it; the row's inputs are
// read after the wait. The state may itself be the previous kernel's output
// (this layer's previous step): the position, read with acquire semantics
// before the copies and again after the wait, tells. It moves only at the
// end of a step, after a release that covers every state write of that
// step, so an unchanged position means the copies saw the state as it is.
// If it moved, the CTA lets its copies land and fetches the state again.
#include <math.h>

#include "o1_common.cuh"

namespace {

__device__ __forceinline__ void tok_wait_primary() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void tok_allow_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ long long tok_ld_acquire(const long long *p) {
    long long v;
    asm volatile("ld.acquire.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ long long tok_ld_relaxed(const long long *p) {
    long long v;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ uint32_t tok_ld_relaxed_u32(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void tok_st_release(long long *p, long long v) {
    asm volatile("st.release.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Bulk copies into shared memory completing on one mbarrier: thread 0 adds
// each copy's bytes and issues it, then arrives once.
__device__ __forceinline__ uint32_t tok_su32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void tok_bulk(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    if (!bytes) return;
    asm volatile("mbarrier.expect_tx.shared::cta.b64 [%0], %1;" ::"r"(tok_su32(bar)), "r"(bytes) : "memory");
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     tok_su32(dst)),
                 "l"((uint64_t)src), "r"(bytes), "r"(tok_su32(bar))
                 : "memory");
}
__device__ __forceinline__ void tok_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tok_su32(bar)) : "memory");
}
__device__ __forceinline__ bool tok_wait(uint64_t *bar, uint32_t parity, long long limit) {
    const long long t0 = clock64();
    while (true) {
        uint32_t ok;
        asm volatile(
            "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(ok)
            : "r"(tok_su32(bar)), "r"(parity)
            : "memory");
        if (ok) return true;
        if (clock64() - t0 > limit) return false;
    }
}
// Waits for the block's copies (limit a.wait_cycles); on expiry raises the
// flag and waits once more, with the full limit, for the copies still in
// flight (they write this block's shared memory), then carries on.
__device__ __forceinline__ void tok_wait_copies(const O1Args &a, uint64_t *bar, uint32_t parity) {
    if (!tok_wait(bar, parity, a.wait_cycles)) {
        if (threadIdx.x == 0) atomicOr(&a.hdr->flags, (uint32_t)O1_FLAG_WAIT_EXPIRED);
        tok_wait(bar, parity, O1_WAIT_CYCLES_FULL);
    }
}

// Rotary angle of pair j at the row's position (identity when the layer
// does not rotate).
__device__ __forceinline__ void tok_cs(const O1Args &a, float inv, long long p, float &cs, float &sn) {
    cs = 1.f;
    sn = 0.f;
    if (a.rotate) o1_rope_cs(inv, p, cs, sn);
}

// Dot products of shared-memory rows (d floats each) with `nq` vectors (d
// floats, `qstride` apart), lane = row, warp = a contiguous share of d in
// float4 units (U = d / 32 of them, at most 8), visited from a lane-dependent
// start so that the lanes of a quarter warp read different bank groups.
// Returns the warp's partial dots in acc[0 .. nq-1] (0 for an invalid row).
// A runtime loop over the warp's units keeps the code short: the kernel is
// latency-bound and its instruction fetch shows.
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
    int sidx = lane % U;
#pragma unroll 2
    for (int t = 0; t < U; ++t) {
        const int u = ub + sidx;
        if (++sidx == U) sidx = 0;
        if (u >= nu) continue;
        const float4 kv = kr[u];
#pragma unroll
        for (int h = 0; h < NQ; ++h) {
            if (h >= nq) break;
            const float4 qv = ((const float4 *)(qs + (size_t)h * qstride))[u];
            acc[h] = fmaf(qv.x, kv.x, fmaf(qv.y, kv.y, fmaf(qv.z, kv.z, fmaf(qv.w, kv.w, acc[h]))));
        }
    }
}

// The same for one vector, its units held in registers: Q.q[t] is unit
// ub + (lane % U + t) % U of the vector, the unit tok_dot1 reads of a row at
// step t, so that a row costs one shared-memory load per unit.
struct TokQ1 {
    float4 q[8];
};
__device__ __forceinline__ void tok_q1_load(const float *qs, int d, TokQ1 &Q) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nu = d >> 2, U = (nu + 7) >> 3, ub = warp * U;
    int sidx = lane % U;
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        const int u = ub + sidx;
        Q.q[t] = (t < U && u < nu) ? ((const float4 *)qs)[u] : make_float4(0.f, 0.f, 0.f, 0.f);
        if (++sidx == U) sidx = 0;
    }
}
__device__ __forceinline__ float tok_dot1(const float *rows, int row, bool valid, const TokQ1 &Q, int d) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nu = d >> 2, U = (nu + 7) >> 3, ub = warp * U;
    if (!valid) return 0.f;
    const float4 *kr = (const float4 *)(rows + (size_t)row * d);
    int sidx = lane % U;
    float acc = 0.f;
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        if (t >= U) break;
        const int u = ub + sidx;
        if (++sidx == U) sidx = 0;
        if (u < nu) {
            const float4 kv = kr[u];
            acc = fmaf(Q.q[t].x, kv.x, fmaf(Q.q[t].y, kv.y, fmaf(Q.q[t].z, kv.z, fmaf(Q.q[t].w, kv.w, acc))));
        }
    }
    return acc;
}

// What a CTA of the step is.
struct TokRole {
    bool far;
    int g, h, hl, fc, c;
};

__device__ __forceinline__ TokRole tok_role(const O1Args &a) {
    TokRole r;
    const int nfar = a.nh * a.NF, bx = blockIdx.x;
    if (bx < nfar) {   // far chunks first: theirs is the longer chain
        r.far = true;
        r.h = bx / a.NF;
        r.fc = bx - r.h * a.NF;
        r.g = r.h / a.hpg;
        r.hl = r.h - r.g * a.hpg;
        r.c = 0;
    } else {
        const int i = bx - nfar;
        r.far = false;
        r.g = i / a.NC;
        r.c = i - r.g * a.NC;
        r.h = r.hl = r.fc = 0;
    }
    return r;
}

// The group's near set after the push, and a slice of it.
struct TokNear {
    bool evict;
    int len1, head1, n, i0, cnt;
    int ipush;   // the slice's index of the pushed key (the near set's last), or -1
};

__device__ __forceinline__ TokNear tok_near_plan(const O1Args &a, const O1Meta &mt, int c) {
    TokNear p;
    p.evict = mt.len0 == mt.wg;
    p.len1 = p.evict ? mt.wg : mt.len0 + 1;
    p.head1 = p.evict ? (mt.head0 + 1) % mt.wg : mt.head0;
    p.n = a.ns + p.len1;
    p.i0 = c * a.KC;
    p.cnt = max(0, min(a.KC, p.n - p.i0));
    p.ipush = (p.cnt > 0 && p.i0 + p.cnt == p.n) ? p.cnt - 1 : -1;
    return p;
}

// Shared memory of a near slice (floats; the offsets o1_tok_near_floats sums).
struct TokNearSm {
    uint64_t *bar;
    float *sq, *sk, *svr, *sgt, *sK, *sV, *sS, *sP, *smg;
};
__device__ __forceinline__ TokNearSm tok_near_sm(const O1Args &a, float *sm) {
    TokNearSm s;
    s.bar = (uint64_t *)sm;
    s.sq = sm + 4;                          // [hpg][d]   rotated queries
    s.sk = s.sq + a.hpg * a.d;              // [d]        the row's rotated key
    s.svr = s.sk + a.d;                     // [dv]       the row's value
    s.sgt = s.svr + a.dv;                   // [hpg][dv]  gate logits (for a merge)
    s.sK = s.sgt + a.hpg * a.dv;            // [KC][d]
    s.sV = s.sK + (size_t)a.KC * a.d;       // [KC][dv]
    s.sS = s.sV + (size_t)a.KC * a.dv;      // [KC][hpg]  scores, then weights
    s.sP = s.sS + (size_t)a.KC * a.hpg;     // [8][KC][hpg] partial dots
    // the merge's staging reuses sK onwards; the merge scratch follows it
    const size_t r = o1_tok_near_region(a.d, a.dv, a.hpg, a.KC), st = o1_tok_stage_min(a.hpg, a.NC, a.NF, a.dv);
    s.smg = s.sK + (r > st ? r : st);
    return s;
}

// Shared memory of a far chunk (floats; o1_tok_far_floats).
struct TokFarSm {
    uint64_t *bar;
    float *sq, *sk, *ske, *svr, *sve, *sgt, *sqt, *skt, *sT, *smu, *sPf, *sPl, *sF, *sG, *sRho, *sE, *sMn, *sZh,
        *sZl, *sNum, *smg;
};
__device__ __forceinline__ TokFarSm tok_far_sm(const O1Args &a, float *sm) {
    TokFarSm s;
    const int d = a.d, dv = a.dv, m = a.m, MB = a.MB;
    s.bar = (uint64_t *)sm;
    s.sq = sm + 4;                          // [d]       rotated query of the head
    s.sk = s.sq + d;                        // [d]       the row's rotated key
    s.ske = s.sk + d;                       // [d]       the evicted key
    s.svr = s.ske + d;                      // [dv]      the row's value
    s.sve = s.svr + dv;                     // [dv]      the evicted value
    s.sgt = s.sve + dv;                     // [hpg][dv] gate logits (for a merge)
    s.sqt = s.sgt + a.hpg * dv;             // [MB][d]   landmark queries of the chunk
    s.skt = s.sqt + (size_t)MB * d;         // [m][d]    landmark keys of the group
    s.sT = s.skt + (size_t)m * d;           // [MB][dv]  far value sums of the chunk
    s.smu = s.sT + (size_t)MB * dv;         // [m][MB]   mu columns of the chunk
    s.sPf = s.smu + (size_t)m * MB;         // [8][m]    partial dots kt . q'
    s.sPl = s.sPf + 8 * m;                  // [8][MB]   partial dots qt . k_e, then partial u
    s.sF = s.sPl + 8 * MB;                  // [m]       e^{f - F}
    s.sG = s.sF + 2 * m;                    // [MB]      gains
    s.sRho = s.sG + MB;                     // [MB]      rescale of the insert
    s.sE = s.sRho + MB;                     // [MB]      the evicted key's weight
    s.sMn = s.sE + MB;                      // [MB]      far max after the insert
    s.sZh = s.sMn + MB;                     // [MB]      far mass after the insert, high part
    s.sZl = s.sZh + MB;                     // [MB]      and low part
    s.sNum = s.sG + 8 * MB;                 // [256]     numerator partials
    // the merge's staging reuses sqt onwards; the merge scratch follows it,
    // 16-byte aligned
    const size_t r = o1_tok_far_region(d, dv, m, MB), st = o1_tok_stage_min(a.hpg, a.NC, a.NF, dv);
    s.smg = (float *)(((uintptr_t)(s.sqt + (r > st ? r : st)) + 15) & ~(uintptr_t)15);
    return s;
}

// Thread 0: the copies of the state a CTA needs, for meta `mt`.
template <bool CO>
__device__ void tok_issue(const O1Args &a, const TokRole &ro, const O1Meta &mt, float *sm) {
    const int d = a.d, dv = a.dv;
    if (!ro.far) {
        const TokNearSm s = tok_near_sm(a, sm);
        const TokNear p = tok_near_plan(a, mt, ro.c);
        // sinks, then ring logical indices as at most two contiguous runs
        // (to the ring's end, from slot 0), one bulk copy each for K and V.
        // The pushed key (the near set's last, always a ring key) is not
        // copied: this row overwrites its slot, and tok_inputs_finish puts
        // the row's own rotated key and value in its place.
        const int ccopy = p.ipush >= 0 ? p.cnt - 1 : p.cnt;
        const int nsk = max(0, min(ccopy, a.ns - p.i0));
        if (nsk > 0) {
            tok_bulk(s.sK, a.sink_k + ((size_t)ro.g * a.ns + p.i0) * d, (uint32_t)nsk * d * 4, s.bar);
            tok_bulk(s.sV, a.sink_v + ((size_t)ro.g * a.ns + p.i0) * dv, (uint32_t)nsk * dv * 4, s.bar);
        }
        const int nr = ccopy - nsk;
        if (nr > 0) {
            const int L0 = p.i0 + nsk - a.ns;
            const int s0 = (p.head1 + L0) % mt.wg;
            const int na = min(nr, mt.wg - s0);
            tok_bulk(s.sK + (size_t)nsk * d, a.ring_k + ((size_t)ro.g * a.w + s0) * d, (uint32_t)na * d * 4, s.bar);
            tok_bulk(s.sV + (size_t)nsk * dv, a.ring_v + ((size_t)ro.g * a.w + s0) * dv, (uint32_t)na * dv * 4, s.bar);
            if (nr > na) {
                tok_bulk(s.sK + (size_t)(nsk + na) * d, a.ring_k + (size_t)ro.g * a.w * d, (uint32_t)(nr - na) * d * 4,
                         s.bar);
                tok_bulk(s.sV + (size_t)(nsk + na) * dv, a.ring_v + (size_t)ro.g * a.w * dv,
                         (uint32_t)(nr - na) * dv * 4, s.bar);
            }
        }
    } else if constexpr (CO) {
        // the insert's operands only: landmark queries, T rows, the evicted pair
        const TokFarSm s = tok_far_sm(a, sm);
        const int b0 = ro.fc * a.MB, nb = max(0, min(a.MB, a.m - b0));
        if (mt.len0 == mt.wg && nb > 0) {
            tok_bulk(s.sT, a.T + ((size_t)ro.h * a.m + b0) * dv, (uint32_t)nb * dv * 4, s.bar);
            tok_bulk(s.sqt, a.qt + ((size_t)ro.h * a.m + b0) * d, (uint32_t)nb * d * 4, s.bar);
            tok_bulk(s.ske, a.ring_k + ((size_t)ro.g * a.w + mt.head0) * d, (uint32_t)d * 4, s.bar);
            tok_bulk(s.sve, a.ring_v + ((size_t)ro.g * a.w + mt.head0) * dv, (uint32_t)dv * 4, s.bar);
        }
    } else {
        const TokFarSm s = tok_far_sm(a, sm);
        const bool evict = mt.len0 == mt.wg;
        const int farl1 = mt.farl0 + (evict ? 1 : 0);
        const int b0 = ro.fc * a.MB, nb = max(0, min(a.MB, a.m - b0));
        if (farl1 > 0 && nb > 0) {
            tok_bulk(s.skt, a.kt + (size_t)ro.g * a.m * d, (uint32_t)a.m * d * 4, s.bar);
            tok_bulk(s.sT, a.T + ((size_t)ro.h * a.m + b0) * dv, (uint32_t)nb * dv * 4, s.bar);
            if (evict) {
                tok_bulk(s.sqt, a.qt + ((size_t)ro.h * a.m + b0) * d, (uint32_t)nb * d * 4, s.bar);
                tok_bulk(s.ske, a.ring_k + ((size_t)ro.g * a.w + mt.head0) * d, (uint32_t)d * 4, s.bar);
                tok_bulk(s.sve, a.ring_v + ((size_t)ro.g * a.w + mt.head0) * dv, (uint32_t)dv * 4, s.bar);
            }
        }
    }
    tok_arrive((uint64_t *)sm);
}

// 16-byte asynchronous global -> shared copies (the row's value and gate
// logits), completed by tok_cp_wait.
__device__ __forceinline__ void tok_cp16(float *dst, const float *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(tok_su32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void tok_cp_wait() {
    asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;" ::: "memory");
}

// The row's inputs a CTA of group g holds: its rotated key and value (for
// the push and the commit), the gate logits of the group's heads (for a
// merge), and the rotated queries of `nq` heads from head q0. Issued right
// after the wait (tok_inputs_load), finished once the position is known.
template <int HPG>
struct TokIn {
    float x0[HPG + 1], x1[HPG + 1];
};
template <int HPG>
__device__ __forceinline__ void tok_inputs_load(const O1Args &a, int g, int q0, int nq, TokIn<HPG> &in, float *svr,
                                                float *sgt) {
    const int tid = threadIdx.x, d = a.d, dv = a.dv, half = d >> 1;
    const bool rj = tid < half;
#pragma unroll
    for (int h = 0; h <= HPG; ++h) {
        const float *src = h < nq ? a.q + (size_t)(q0 + h) * d : a.k + (size_t)g * d;
        const bool ok = rj && h <= nq;
        in.x0[h] = ok ? src[tid] : 0.f;
        in.x1[h] = ok ? src[tid + half] : 0.f;
    }
    for (int t = tid; t < (dv >> 2); t += blockDim.x) tok_cp16(svr + 4 * t, a.v + (size_t)g * dv + 4 * t);
    if (a.gate)
        for (int t = tid; t < ((a.hpg * dv) >> 2); t += blockDim.x)
            tok_cp16(sgt + 4 * t, a.gate + (size_t)g * a.hpg * dv + 4 * t);
}
// A near slice holding the pushed key gets the row's rotated key and value
// in that key's place (kpush, vpush; null otherwise). Called after the
// copies of a stale prefetch have landed, so that none overwrites them.
template <int HPG>
__device__ __forceinline__ void tok_inputs_finish(const O1Args &a, int g, int nq, float cs, float sn,
                                                  const TokIn<HPG> &in, float *sq, float *sk, float *kpush,
                                                  float *vpush) {
    const int tid = threadIdx.x, d = a.d, half = d >> 1;
    if (tid < half) {
#pragma unroll
        for (int h = 0; h <= HPG; ++h) {
            if (h > nq) break;
            float *dst = h < nq ? sq + h * d : sk;
            const float y0 = in.x0[h] * cs - in.x1[h] * sn, y1 = in.x1[h] * cs + in.x0[h] * sn;
            dst[tid] = y0;
            dst[tid + half] = y1;
            if (h == nq && kpush) {
                kpush[tid] = y0;
                kpush[tid + half] = y1;
            }
        }
    }
    if (vpush)
        for (int t = tid; t < (a.dv >> 2); t += blockDim.x) tok_cp16(vpush + 4 * t, a.v + (size_t)g * a.dv + 4 * t);
}

// A near slice for up to 4 heads a group: lanes across the vectors' columns
// (the queries in registers, each key row read once and without bank
// conflicts), warps across keys (key = warp + 8 i). A warp's per-lane partial
// dots leave it through one reduce-scatter (warp_reduce_scatter32): lane l
// ends with the sum of value l, value i HPG + h being key i's score for head h.
// The value sums go the same way round (warps across keys, lanes across
// columns, every head in registers); the 8 warps' partials meet in the key
// rows' shared memory, free by then.
template <int HPG>
__device__ void tok_near_small(const O1Args &a, const TokNearSm &s, int cnt, float *pv, float *pml, size_t hs) {
    static_assert(HPG <= 4, "registers hold HPG queries and HPG value sums");
    constexpr int KPB = 32 / HPG;   // a warp's keys per butterfly
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int hpg = a.hpg, nu = a.d >> 2, nv = a.dv >> 2;   // float4 units of a key, of a value (<= 64)
    const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
    const float4 *sq4 = (const float4 *)s.sq, *sK4 = (const float4 *)s.sK, *sV4 = (const float4 *)s.sV;
    float4 qr[HPG][2];
#pragma unroll
    for (int h = 0; h < HPG; ++h)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int u = lane + 32 * j;
            qr[h][j] = (h < hpg && u < nu) ? sq4[h * nu + u] : z4;
        }
    const int kpw = (cnt + 7) >> 3;   // keys of the busiest warp
    for (int i0 = 0; i0 < kpw; i0 += KPB) {
        float x[32];
#pragma unroll
        for (int i = 0; i < KPB; ++i) {
            const int key = warp + 8 * (i0 + i);
            float4 k0 = z4, k1 = z4;
            if (key < cnt) {
                if (lane < nu) k0 = sK4[(size_t)key * nu + lane];
                if (lane + 32 < nu) k1 = sK4[(size_t)key * nu + lane + 32];
            }
#pragma unroll
            for (int h = 0; h < HPG; ++h) {
                float acc = qr[h][0].x * k0.x;
                acc = fmaf(qr[h][0].y, k0.y, acc);
                acc = fmaf(qr[h][0].z, k0.z, acc);
                acc = fmaf(qr[h][0].w, k0.w, acc);
                acc = fmaf(qr[h][1].x, k1.x, acc);
                acc = fmaf(qr[h][1].y, k1.y, acc);
                acc = fmaf(qr[h][1].z, k1.z, acc);
                acc = fmaf(qr[h][1].w, k1.w, acc);
                x[i * HPG + h] = acc;
            }
        }
#pragma unroll
        for (int i = KPB * HPG; i < 32; ++i) x[i] = 0.f;
        warp_reduce_scatter32(x);
        const int i = lane / HPG, h = lane - i * HPG, key = warp + 8 * (i0 + i);
        if (i < KPB && h < hpg && key < cnt) s.sS[key * hpg + h] = x[0] * a.scale;
    }
    __syncthreads();
    // per head (a warp each): the slice max, the weights e^{s - max} and their sum
    for (int h = warp; h < hpg; h += 8) {
        float mx = -INFINITY;
        for (int i = lane; i < cnt; i += 32) mx = fmaxf(mx, s.sS[i * hpg + h]);
        mx = warp_max(mx);
        float l = 0.f;
        for (int i = lane; i < cnt; i += 32) {
            const float e = expf(s.sS[i * hpg + h] - mx);
            s.sS[i * hpg + h] = e;
            l += e;
        }
        l = warp_sum(l);
        if (lane == 0) {
            pml[h * hs * 2] = mx;
            pml[h * hs * 2 + 1] = l;
        }
    }
    __syncthreads();
    float4 acc[HPG][2];
#pragma unroll
    for (int h = 0; h < HPG; ++h) acc[h][0] = acc[h][1] = z4;
    for (int key = warp; key < cnt; key += 8) {
        float w[HPG];
#pragma unroll
        for (int h = 0; h < HPG; ++h) w[h] = h < hpg ? s.sS[key * hpg + h] : 0.f;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int c = lane + 32 * j;
            if (c >= nv) continue;
            const float4 v = sV4[(size_t)key * nv + c];
#pragma unroll
            for (int h = 0; h < HPG; ++h) {
                acc[h][j].x = fmaf(w[h], v.x, acc[h][j].x);
                acc[h][j].y = fmaf(w[h], v.y, acc[h][j].y);
                acc[h][j].z = fmaf(w[h], v.z, acc[h][j].z);
                acc[h][j].w = fmaf(w[h], v.w, acc[h][j].w);
            }
        }
    }
    __syncthreads();   // every warp is done with the key and value rows
    float4 *red = (float4 *)s.sK;   // [8][hpg][nv]: 8 hpg dv floats fit (o1_tok_near_floats)
#pragma unroll
    for (int h = 0; h < HPG; ++h)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int c = lane + 32 * j;
            if (h < hpg && c < nv) red[((size_t)warp * hpg + h) * nv + c] = acc[h][j];
        }
    __syncthreads();
    for (int idx = tid; idx < hpg * nv; idx += blockDim.x) {
        const int h = idx / nv, c = idx - h * nv;
        float4 t = red[(size_t)h * nv + c];
#pragma unroll
        for (int w = 1; w < 8; ++w) {
            const float4 o = red[((size_t)w * hpg + h) * nv + c];
            t.x += o.x;
            t.y += o.y;
            t.z += o.z;
            t.w += o.w;
        }
        ((float4 *)(pv + h * hs * a.dv))[c] = t;
    }
}

// A near slice: scores of every head of the group over the slice's keys, a
// slice-local softmax and the value sums -> partial (max, sum, value sum).
template <int HPG>
__device__ void tok_near_compute(const O1Args &a, const TokRole &ro, const O1Meta &mt, const TokNearSm &s) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int d = a.d, dv = a.dv, hpg = a.hpg, KC = a.KC;
    const TokNear p = tok_near_plan(a, mt, ro.c);
    const int cnt = p.cnt;
    // head h's partial: pv + h NC dv (value sums), pml + h NC 2 (max, sum)
    const size_t slot = (size_t)ro.g * hpg * a.NC + ro.c, hs = (size_t)a.NC;
    float *pv = a.part + slot * dv;
    float *pml = a.pml + slot * 2;
    if (ro.c == 0)   // the group's rotated key, for the commit
        for (int j = tid; j < d; j += blockDim.x) a.kcur[(size_t)ro.g * d + j] = s.sk[j];
    if (cnt == 0) {   // an empty slice: zero weight, and zero sums (the merge reads every row)
        for (int h = tid; h < hpg; h += blockDim.x) {
            pml[h * hs * 2] = -INFINITY;
            pml[h * hs * 2 + 1] = 0.f;
        }
        const int dv4 = dv >> 2;
        for (int i = tid; i < hpg * dv4; i += blockDim.x) {
            const int h = i / dv4;
            ((float4 *)(pv + h * hs * dv))[i - h * dv4] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        return;
    }
    // (the pushed key's row holds the row's own rotated key and value)
    if constexpr (HPG <= 4) {
        tok_near_small<HPG>(a, s, cnt, pv, pml, hs);
    } else {
        // scores: partial dots per warp (lane = key) over the warp's share of d
        for (int k0 = 0; k0 < cnt; k0 += 32) {
            float acc[HPG];
            const int key = k0 + lane;
            tok_dots(s.sK, key, key < cnt, s.sq, d, hpg, d, acc);
            if (key < cnt)
#pragma unroll
                for (int h = 0; h < HPG; ++h) {
                    if (h >= hpg) break;
                    s.sP[((size_t)warp * KC + key) * hpg + h] = acc[h];
                }
        }
        __syncthreads();
        // per head (a warp each): the partials' sums and the slice max, then the
        // weights e^{s - max} and their sum
        for (int h = warp; h < hpg; h += blockDim.x >> 5) {
            float mx = -INFINITY;
            for (int i = lane; i < cnt; i += 32) {
                float acc = 0.f;
#pragma unroll
                for (int w = 0; w < 8; ++w) acc += s.sP[((size_t)w * KC + i) * hpg + h];
                acc *= a.scale;
                s.sS[i * hpg + h] = acc;
                mx = fmaxf(mx, acc);
            }
            mx = warp_max(mx);
            float l = 0.f;
            for (int i = lane; i < cnt; i += 32) {
                const float e = expf(s.sS[i * hpg + h] - mx);
                s.sS[i * hpg + h] = e;
                l += e;
            }
            l = warp_sum(l);
            if (lane == 0) {
                pml[h * hs * 2] = mx;
                pml[h * hs * 2 + 1] = l;
            }
        }
        __syncthreads();
        // value sums: thread per (head, 4 columns)
        const int dv4 = dv >> 2;
        for (int idx = tid; idx < hpg * dv4; idx += blockDim.x) {
            const int h = idx / dv4, c4 = idx - h * dv4;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
            for (int i = 0; i < cnt; ++i) {
                const float w = s.sS[i * hpg + h];
                const float4 v = ((const float4 *)(s.sV + (size_t)i * dv))[c4];
                acc.x = fmaf(w, v.x, acc.x);
                acc.y = fmaf(w, v.y, acc.y);
                acc.z = fmaf(w, v.z, acc.z);
                acc.w = fmaf(w, v.w, acc.w);
            }
            ((float4 *)(pv + h * hs * dv))[c4] = acc;
        }
    }
}

// A far chunk: landmark queries b in [b0, b0 + nb) of head h. The insert of
// the evicted key (o1b_far_e / o1b_far_commit for one row): l_b, M' =
// max(M, l_b), rho, e, Z (in float-float, high and low parts), T; then the
// readout's share: F and e^{f - F} over every landmark key, u_b, the chunk's
// exponent c_f = max_b (F + M'_b), gains, the chunk's far mass (float-float) and
// numerator -> the far record (c_f, D, numerator), all relative to c_f.
// Warp 1, lane b, holds the chunk's entering M and Z (Mo, Zo).
__device__ void tok_far_compute(const O1Args &a, const TokRole &ro, const O1Meta &mt, const TokFarSm &s, float Mo,
                                o1_ff Zo) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int d = a.d, dv = a.dv, m = a.m, MB = a.MB, h = ro.h;
    const bool evict = mt.len0 == mt.wg;
    const int farl1 = mt.farl0 + (evict ? 1 : 0);
    const int b0 = ro.fc * MB, nb = max(0, min(MB, m - b0));
    float *fp = a.farp + ((size_t)h * a.NF + ro.fc) * (4 + dv);
    __shared__ float s_Dh, s_Dl;
    if (farl1 == 0 || nb == 0) {   // no far field, or no landmark here: an empty record
        for (int t = tid; t < dv; t += blockDim.x) fp[4 + t] = 0.f;
        if (tid == 0) {
            fp[0] = -INFINITY;
            fp[2] = fp[3] = 0.f;
        }
        return;
    }
    // partial dots per warp, lane = landmark: kt_a . q' (every a), and
    // qt_b . k_e (the chunk's b, when a key is evicted)
    {
        TokQ1 Q;
        tok_q1_load(s.sq, d, Q);
        for (int a0 = 0; a0 < m; a0 += 32) {
            const int aa = a0 + lane;
            const float f = tok_dot1(s.skt, aa, aa < m, Q, d);
            if (aa < m) s.sPf[warp * m + aa] = f;
        }
        if (evict) tok_q1_load(s.ske, d, Q);
        const float l = tok_dot1(s.sqt, lane, evict && lane < nb, Q, d);
        if (lane < nb) s.sPl[warp * MB + lane] = l;
    }
    __syncthreads();
    // Every warp: F = max_a f_a and e^{f_a - F} for a = lane, lane + 32 (the
    // same in each warp, so that no warp waits for another); then u_b for its
    // share of the chunk's landmarks (b = warp, warp + 8, ...), a warp sum
    // over a each. Warp 1 also takes the insert, lane = b.
    float F;
    {
        float f0 = -INFINITY, f1 = -INFINITY;
        if (lane < m) {
            float acc = 0.f;
#pragma unroll
            for (int w = 0; w < 8; ++w) acc += s.sPf[w * m + lane];
            f0 = acc * a.scale;
        }
        if (lane + 32 < m) {
            float acc = 0.f;
#pragma unroll
            for (int w = 0; w < 8; ++w) acc += s.sPf[w * m + lane + 32];
            f1 = acc * a.scale;
        }
        F = warp_max(fmaxf(f0, f1));
        const float e0 = lane < m ? expf(f0 - F) : 0.f, e1 = lane + 32 < m ? expf(f1 - F) : 0.f;
        for (int b = warp; b < nb; b += 8) {
            float part = 0.f;
            if (lane < m) part = e0 * s.smu[lane * MB + b];
            if (lane + 32 < m) part = fmaf(e1, s.smu[(lane + 32) * MB + b], part);
            float u = warp_sum(part);
            if (a.rect) u = fmaxf(u, 0.f);
            if (lane == 0) s.sG[b] = u;   // u_b here; the gain is formed from it below
        }
    }
    if (warp == 1 && lane < nb) {
        // the insert of the evicted key for landmark query b = b0 + lane
        float Mn = Mo, rho = 1.f, e = 0.f;
        o1_ff Zn = Zo;
        if (evict) {
            float l = 0.f;
#pragma unroll
            for (int w = 0; w < 8; ++w) l += s.sPl[w * MB + lane];
            l *= a.scale;
            Mn = fmaxf(Mo, l);
            rho = (Mn == Mo) ? 1.f : expf(Mo - Mn);
            e = expf(l - Mn);
            Zn = ff_add_f(ff_mul_f(Zo, rho), e);
            const size_t at = (size_t)h * m + b0 + lane;
            a.M[at] = Mn;
            a.Z[at] = Zn.hi;
            a.Zlo[at] = Zn.lo;
        }
        s.sRho[lane] = rho;
        s.sE[lane] = e;
        s.sMn[lane] = Mn;
        s.sZh[lane] = Zn.hi;
        s.sZl[lane] = Zn.lo;
    }
    __syncthreads();
    // Every warp: the chunk's exponent c_f = max_b (F + M'_b). Gains
    // g_b = u_b e^{F + M'_b - c_f}; warp 0 sums the chunk's far mass
    // D = sum_b g_b Z_b in float-float (its terms can cancel to a small
    // fraction of their size); every thread inserts the evicted value into
    // its share of T, writes T back and forms partial far numerators.
    const float cf = warp_max(lane < nb ? F + s.sMn[lane] : -INFINITY);
    if (warp == 0) {
        const float gn = lane < nb ? s.sG[lane] * expf(F + s.sMn[lane] - cf) : 0.f;
        const o1_ff D = warp_sum(lane < nb ? ff_mul_f(ff_make(s.sZh[lane], s.sZl[lane]), gn) : ff_make(0.f, 0.f));
        if (lane == 0) {
            s_Dh = D.hi;
            s_Dl = D.lo;
        }
    }
    const int nlg = blockDim.x / dv, t = tid % dv, lg = tid / dv;
    if (lg < nlg) {
        const float vt = evict ? s.sve[t] : 0.f;
        float acc = 0.f;
        for (int b = lg; b < nb; b += nlg) {
            float x = s.sT[b * dv + t];
            if (evict) {
                x = s.sRho[b] * x + s.sE[b] * vt;
                a.T[((size_t)h * m + b0 + b) * dv + t] = x;
            }
            acc = fmaf(s.sG[b] * expf(F + s.sMn[b] - cf), x, acc);
        }
        s.sNum[lg * dv + t] = acc;
    }
    __syncthreads();
    for (int c = tid; c < dv; c += blockDim.x) {
        float acc = 0.f;
        for (int q = 0; q < nlg; ++q) acc += s.sNum[q * dv + c];
        fp[4 + c] = acc;
    }
    if (tid == 0) {
        fp[0] = cf;
        fp[2] = s_Dh;
        fp[3] = s_Dl;
    }
}

// A pushed row without attention (o1_spec_commit of one row): the far
// chunk's insert of the evicted key only, with the same arithmetic as
// tok_far_compute: l_b, M' = max(M, l_b), rho, e, Z in float-float, and T.
__device__ void tok_far_insert(const O1Args &a, const TokRole &ro, const O1Meta &mt, const TokFarSm &s, float Mo,
                               o1_ff Zo) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int d = a.d, dv = a.dv, m = a.m, MB = a.MB, h = ro.h;
    const int b0 = ro.fc * MB, nb = max(0, min(MB, m - b0));
    if (mt.len0 != mt.wg || nb == 0) return;   // nothing evicted, or no landmark here
    {
        TokQ1 Q;
        tok_q1_load(s.ske, d, Q);
        const float l = tok_dot1(s.sqt, lane, lane < nb, Q, d);
        if (lane < nb) s.sPl[warp * MB + lane] = l;
    }
    __syncthreads();
    if (warp == 1 && lane < nb) {
        float l = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) l += s.sPl[w * MB + lane];
        l *= a.scale;
        const float Mn = fmaxf(Mo, l);
        const float rho = (Mn == Mo) ? 1.f : expf(Mo - Mn);
        const float e = expf(l - Mn);
        const o1_ff Zn = ff_add_f(ff_mul_f(Zo, rho), e);
        const size_t at = (size_t)h * m + b0 + lane;
        a.M[at] = Mn;
        a.Z[at] = Zn.hi;
        a.Zlo[at] = Zn.lo;
        s.sRho[lane] = rho;
        s.sE[lane] = e;
    }
    __syncthreads();
    for (int i = tid; i < nb * dv; i += blockDim.x) {
        const int b = i / dv, t = i - b * dv;
        a.T[((size_t)h * m + b0 + b) * dv + t] = s.sRho[b] * s.sT[b * dv + t] + s.sE[b] * s.sve[t];
    }
}

// Bulk copy without its own expect-tx: the bytes of a batch of them are
// announced once on the barrier (tok_merge_issue).
__device__ __forceinline__ void tok_bulk_nx(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     tok_su32(dst)),
                 "l"((uint64_t)src), "r"(bytes), "r"(tok_su32(bar))
                 : "memory");
}
// Barrier 1 over the first `nthr` threads (the merge's; barrier 0 is the CTA's).
__device__ __forceinline__ void tok_bar_merge(int nthr) { asm volatile("bar.sync 1, %0;" ::"r"(nthr) : "memory"); }
// The si-th head (0-based, in order) of the set `mine`.
__device__ __forceinline__ int tok_nth_head(unsigned mine, int si) {
    for (int k = 0; k < si; ++k) mine &= mine - 1;
    return __ffs(mine) - 1;
}

// One thread: the bulk copies of a merge's round, for every head si of
// `mine`: near rows [r0, r1) of its slices (contiguous in `part`) to
// buf[si][R][dv], and in the first round its NF far records (contiguous in
// `farp`, 4 + dv floats each) to far[si][NF][4 + dv].
__device__ void tok_merge_issue(const O1Args &a, int g, unsigned mine, int nS, int r0, int r1, int R, float *buf,
                                float *far, uint64_t *bar) {
    const int hpg = a.hpg, NC = a.NC, NF = a.NF, dv = a.dv;
    // the data were written by generic stores (other CTAs', ordered before
    // the arrival's acquire) and the buffers last held this CTA's own
    // generic accesses: order both before the async proxy's copies
    asm volatile("fence.proxy.async.global;\nfence.proxy.async.shared::cta;" ::: "memory");
    const uint32_t near_b = (uint32_t)(r1 - r0) * dv * 4, far_b = far ? (uint32_t)NF * (4 + dv) * 4 : 0u;
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(tok_su32(bar)),
                 "r"((uint32_t)nS * (near_b + far_b))
                 : "memory");
    unsigned left = mine;
    for (int si = 0; si < nS; ++si) {
        const int hl = __ffs(left) - 1;
        left &= left - 1;
        tok_bulk_nx(buf + (size_t)si * R * dv, a.part + ((size_t)(g * hpg + hl) * NC + r0) * dv, near_b, bar);
        if (far)
            tok_bulk_nx(far + (size_t)si * NF * (4 + dv), a.farp + (size_t)(g * hpg + hl) * NF * (4 + dv), far_b, bar);
    }
}

// The merge of the heads in `mine` (bits hl of group g), by the CTA that
// arrived last for them, on its first `nthr` threads: per head, the near
// slices' (max, sum) -> the window max M_w and mass L; the far records ->
// c_f and D (float-float, sign decision); then per (head, 4 columns) the
// slices' value sums (each moved to M_w), the far numerator, one exponent
// c = max(M_w, c_f) (the far max counts even when the far part is dropped,
// as the pages' c_all does), the 1e-30 floor and the gate.
// The rows summed come into shared memory by bulk copies (two a head, issued
// by the last warp's first thread): all at once when they fit, else in
// rounds through two buffers; the statistics are formed from global memory
// while the first copies fly. `stage` is shared memory the CTA's own work is
// done with (at least o1_tok_stage_min floats), `shd` the merge scratch,
// `bars` two mbarriers.
template <int HPG>
__device__ void tok_merge(const O1Args &a, int g, unsigned mine, int farl1, const float *sgt, float *shd,
                          float *stage, size_t stage_floats, uint64_t *bars, int nthr) {
    constexpr int MAXP = (HPG * 64 + 223) / 224;   // passes over the (head, 4 columns) items
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = nthr >> 5;
    const int hpg = a.hpg, NC = a.NC, NF = a.NF, dv = a.dv, dv4 = dv >> 2, RT = NC + NF;
    const int nS = __popc(mine);
    const bool issuer = tid == nthr - 32;
    float *fac = stage;   // [nS][RT] row factors
    const size_t ffl = ((size_t)nS * RT + 3) / 4 * 4;
    float *far = stage + ffl;   // [nS][NF][4 + dv]
    float *rows = far + (size_t)nS * NF * (4 + dv);
    const size_t row_floats = (size_t)nS * dv, avail = stage_floats - ffl - (size_t)nS * NF * (4 + dv);
    int nbuf = 1, R = NC;
    if ((size_t)NC * row_floats > avail) {
        R = (int)(avail / (2 * row_floats));
        nbuf = 2;
        if (R < 1) {
            R = (int)(avail / row_floats);
            nbuf = 1;
        }
    }
    const int nr = (NC + R - 1) / R;
    if (issuer)
        for (int k = 0; k < nbuf && k < nr; ++k)
            tok_merge_issue(a, g, mine, nS, k * R, min(NC, (k + 1) * R), R, rows + (size_t)k * R * row_floats,
                            k == 0 ? far : nullptr, bars + k);

    // statistics, a warp per head, from global memory
    for (int si = warp; si < nS; si += nwarps) {
        const int hl = tok_nth_head(mine, si);
        const int h = g * hpg + hl;
        const float *pml = a.pml + (size_t)h * NC * 2;   // slice c: pml[2 c]
        float *fs = fac + (size_t)si * RT;
        // far record headers (c_r, -, D high, D low): NF <= 64
        float4 fr4[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int r = lane + 32 * k;
            fr4[k] = r < NF ? __ldcg((const float4 *)(a.farp + ((size_t)h * NF + r) * (4 + dv)))
                            : make_float4(-INFINITY, 0.f, 0.f, 0.f);
        }
        float mx = -INFINITY, L = 0.f;
        for (int c = lane; c < NC; c += 32) {
            const float2 v = __ldcg((const float2 *)(pml + 2 * c));
            fs[c] = v.x;
            if (v.x == -INFINITY) continue;
            const float mn = fmaxf(mx, v.x);
            L = L * expf(mx - mn) + v.y * expf(v.x - mn);
            mx = mn;
        }
        const float Mw = warp_max(mx);
        const float cf = warp_max(fmaxf(fr4[0].x, fr4[1].x));
        L = warp_sum(mx == -INFINITY ? 0.f : L * expf(mx - Mw));
        for (int c = lane; c < NC; c += 32) {   // the lane's own entries: no sync needed
            const float mc = fs[c];
            fs[c] = mc == -INFINITY ? 0.f : expf(mc - Mw);
        }
        o1_ff D = ff_make(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int r = lane + 32 * k;
            const float fr = (fr4[k].x == -INFINITY) ? 0.f : expf(fr4[k].x - cf);
            if (r < NF) fs[NC + r] = fr;
            D = ff_add(D, ff_mul_f(ff_make(fr4[k].z, fr4[k].w), fr));
        }
        D = warp_sum(D);
        if (lane == 0) {
            const bool have = farl1 > 0 && ff_nonneg(D);
            shd[si * 8 + 0] = Mw;
            shd[si * 8 + 1] = L;
            shd[si * 8 + 2] = farl1 > 0 ? cf : -INFINITY;
            shd[si * 8 + 3] = have ? 1.f : 0.f;
            shd[si * 8 + 4] = have ? D.hi + D.lo : 0.f;
        }
    }
    tok_bar_merge(nthr);

    // rows: a thread per (head, 4 columns) item and slice group sg (lanes
    // that differ in their high bits), summed over the rows of its group
    const int items = nS * dv4;
    int nsg = 1;
    while (nsg < 8 && items * nsg * 2 <= nthr) nsg *= 2;
    const int lpi = 32 / nsg, sg = lane / lpi, ipp = nthr / nsg;
    const int P = (items + ipp - 1) / ipp;
    float4 A[MAXP];
#pragma unroll
    for (int q = 0; q < MAXP; ++q) A[q] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k = 0; k < nr; ++k) {
        const int r0 = k * R, r1 = min(NC, r0 + R), b = k % nbuf;
        tok_wait_copies(a, bars + b, (uint32_t)((k / nbuf) & 1));
        const float4 *buf = (const float4 *)(rows + (size_t)b * R * row_floats);
#pragma unroll
        for (int q = 0; q < MAXP; ++q) {
            if (q >= P) break;
            const int it = q * ipp + warp * lpi + (lane % lpi);
            if (it >= items) continue;
            const int si = it / dv4, c4 = it - si * dv4;
            const float *fs = fac + (size_t)si * RT;
            const float4 *src = buf + (size_t)si * R * dv4 + c4;
            float4 acc = A[q];
            for (int j = r0 + sg; j < r1; j += nsg) {
                const float f = fs[j];
                const float4 v = src[(size_t)(j - r0) * dv4];
                acc.x = fmaf(f, v.x, acc.x);
                acc.y = fmaf(f, v.y, acc.y);
                acc.z = fmaf(f, v.z, acc.z);
                acc.w = fmaf(f, v.w, acc.w);
            }
            A[q] = acc;
        }
        if (k + nbuf < nr) {   // every thread is done with buffer b: refill it
            tok_bar_merge(nthr);
            if (issuer)
                tok_merge_issue(a, g, mine, nS, (k + nbuf) * R, min(NC, (k + nbuf + 1) * R), R,
                                rows + (size_t)b * R * row_floats, nullptr, bars + b);
        }
    }
    // the far numerators (staged with the first round), the slice groups ->
    // lane sg = 0, then the output
    const int rs4 = (4 + dv) >> 2;
#pragma unroll
    for (int q = 0; q < MAXP; ++q) {
        if (q >= P) break;
        const int it = q * ipp + warp * lpi + (lane % lpi);
        float4 FN = make_float4(0.f, 0.f, 0.f, 0.f);
        if (it < items) {
            const int si = it / dv4, c4 = it - si * dv4;
            const float *fs = fac + (size_t)si * RT + NC;
            const float4 *src = (const float4 *)far + (size_t)si * NF * rs4 + 1 + c4;
            for (int r = sg; r < NF; r += nsg) {
                const float f = fs[r];
                const float4 v = src[(size_t)r * rs4];
                FN.x = fmaf(f, v.x, FN.x);
                FN.y = fmaf(f, v.y, FN.y);
                FN.z = fmaf(f, v.z, FN.z);
                FN.w = fmaf(f, v.w, FN.w);
            }
        }
        for (int off = 16; off >= lpi; off >>= 1) {
            A[q].x += __shfl_xor_sync(0xffffffffu, A[q].x, off);
            A[q].y += __shfl_xor_sync(0xffffffffu, A[q].y, off);
            A[q].z += __shfl_xor_sync(0xffffffffu, A[q].z, off);
            A[q].w += __shfl_xor_sync(0xffffffffu, A[q].w, off);
            FN.x += __shfl_xor_sync(0xffffffffu, FN.x, off);
            FN.y += __shfl_xor_sync(0xffffffffu, FN.y, off);
            FN.z += __shfl_xor_sync(0xffffffffu, FN.z, off);
            FN.w += __shfl_xor_sync(0xffffffffu, FN.w, off);
        }
        if (sg != 0 || it >= items) continue;
        const int si = it / dv4, c4 = it - si * dv4;
        const int hl = tok_nth_head(mine, si), h = g * hpg + hl;
        const float Mw = shd[si * 8 + 0], L = shd[si * 8 + 1], cf = shd[si * 8 + 2];
        const bool have = shd[si * 8 + 3] > 0.5f;
        const float c = cf > -INFINITY ? fmaxf(Mw, cf) : Mw;
        const float al = expf(Mw - c);
        const float be = have ? expf(cf - c) : 0.f;
        const float rden = 1.f / fmaxf(be * shd[si * 8 + 4] + al * L, 1e-30f);
        float y[4] = {(be * FN.x + al * A[q].x) * rden, (be * FN.y + al * A[q].y) * rden,
                      (be * FN.z + al * A[q].z) * rden, (be * FN.w + al * A[q].w) * rden};
        if (a.gate)
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) y[jj] = y[jj] / (1.f + expf(-sgt[hl * dv + 4 * c4 + jj]));
        *((float4 *)(a.out + (size_t)h * dv) + c4) = make_float4(y[0], y[1], y[2], y[3]);
    }
}

// The commit of the step, by one warp of the CTA that arrived last of all
// (every CTA has read the ring, meta and far state by then): each group's
// ring slot gets the row's rotated key and value and its meta moves
// (o1b_ring_commit / o1b_meta for one row); then the position, the step's
// last write, released after every state write of the step. The values and
// the metas are read in one round; `sslot` holds a slot index per group.
__device__ void tok_commit_warp(const O1Args &a, long long p, int *sslot) {
    const int lane = threadIdx.x & 31, G = a.G, d4 = a.d >> 2, dv4 = a.dv >> 2;
    const int nk = G * d4, nt = nk + G * dv4;
    const float4 *kc4 = (const float4 *)a.kcur, *v4 = (const float4 *)a.v;
    float4 *rk4 = (float4 *)a.ring_k, *rv4 = (float4 *)a.ring_v;
    for (int base = 0; base < nt; base += 32 * 8) {
        float4 x[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = base + 32 * u + lane;
            x[u] = i < nk ? __ldcg(kc4 + i) : (i < nt ? __ldcg(v4 + (i - nk)) : make_float4(0.f, 0.f, 0.f, 0.f));
        }
        if (base == 0) {
            for (int g = lane; g < G; g += 32) {
                const int len0 = (int)tok_ld_relaxed_u32(a.meta + g * 4 + 0);
                const int head0 = (int)tok_ld_relaxed_u32(a.meta + g * 4 + 1);
                const int farl0 = (int)tok_ld_relaxed_u32(a.meta + g * 4 + 2);
                const int wg = (int)tok_ld_relaxed_u32(a.meta + g * 4 + 3);
                sslot[g] = (head0 + len0) % wg;
                if (len0 == wg) {
                    a.meta[g * 4 + 1] = (uint32_t)((head0 + 1) % wg);
                    a.meta[g * 4 + 2] = (uint32_t)(farl0 + 1);
                } else {
                    a.meta[g * 4 + 0] = (uint32_t)(len0 + 1);
                }
            }
            __syncwarp();
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = base + 32 * u + lane;
            if (i < nk) {
                const int g = i / d4, j = i - g * d4;
                rk4[((size_t)g * a.w + sslot[g]) * d4 + j] = x[u];
            } else if (i < nt) {
                const int i2 = i - nk, g = i2 / dv4, j = i2 - g * dv4;
                rv4[((size_t)g * a.w + sslot[g]) * dv4 + j] = x[u];
            }
        }
    }
    __syncwarp();
    if (lane == 0) {
        a.tick[a.nh + a.G] = 0u;
        __threadfence();
        tok_st_release((long long *)&a.hdr->pos, p + 1);
    }
}

}  // namespace

// CO: a pushed row without attention (o1_spec_commit of one row): only the
// far chunks, which insert the evicted key; the last CTA commits. A
// separate instance, so that the attending kernel's code does not carry it.
template <int HPG, bool CO>
__global__ __launch_bounds__(256, 2) void k_tok(O1Args a) {
    extern __shared__ __align__(16) float sm[];
    __shared__ long long s_pos;
    __shared__ int s_meta[4];
    __shared__ int s_parity;
    __shared__ unsigned s_mine;
    __shared__ int s_last;
    __shared__ uint64_t s_mbar[2];   // the merge's copies
    const TokRole ro = tok_role(a);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint64_t *bar = (uint64_t *)sm;
    const TokNearSm ns = tok_near_sm(a, sm);
    const TokFarSm fs = tok_far_sm(a, sm);
    float *sq = ro.far ? fs.sq : ns.sq;
    float *sk = ro.far ? fs.sk : ns.sk;
    float *svr = ro.far ? fs.svr : ns.svr;
    float *sgt = ro.far ? fs.sgt : ns.sgt;
    float *smg = ro.far ? fs.smg : ns.smg;

    // ---- before waiting on the previous kernel: this layer's state and
    // constants only
    if (tid == 0) {
        const long long p0 = tok_ld_acquire((const long long *)&a.hdr->pos);
        for (int i = 0; i < 4; ++i) s_meta[i] = (int)tok_ld_relaxed_u32(a.meta + ro.g * 4 + i);
        s_pos = p0;
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(tok_su32(bar)) : "memory");
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(tok_su32(&s_mbar[0])) : "memory");
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(tok_su32(&s_mbar[1])) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        if (a.tok_prefetch) {
            // the copies read global memory through the async proxy: order
            // them after the acquire above
            asm volatile("fence.proxy.async.global;" ::: "memory");
            O1Meta mt;
            mt.len0 = s_meta[0];
            mt.head0 = s_meta[1];
            mt.farl0 = s_meta[2];
            mt.wg = s_meta[3];
            tok_issue<CO>(a, ro, mt, sm);
        }
    }
    const float inv = tid < (a.d >> 1) ? a.hdr->inv_freq[tid] : 0.f;   // a constant of the layer
    if (ro.far && !CO) {   // mu's columns of the chunk: a constant of the layer
        const int b0 = ro.fc * a.MB, nb = max(0, min(a.MB, a.m - b0));
        for (int i = tid; i < a.m * nb; i += blockDim.x) {
            const int aa = i / nb, j = i - aa * nb;
            fs.smu[aa * a.MB + j] = a.mu[((size_t)ro.h * a.m + aa) * a.m + b0 + j];
        }
    }
    __syncthreads();   // the barrier is initialised, the meta snapshot shared
    // the rotation at the position this step most likely runs at: the one
    // read now, or the next one if the previous step on this stream was this
    // layer's (it moves the position at its very end)
    const long long pguess = s_pos + (a.tok_prefetch ? 0 : 1);
    float cs = 1.f, sn = 0.f;
    if (tid < (a.d >> 1)) tok_cs(a, inv, pguess, cs, sn);

    // ---- the previous kernel is done: its outputs (this row) are visible.
    // The row's inputs and the position check go out in one round.
    tok_wait_primary();
    tok_allow_dependents();
    TokIn<HPG> in;
    if (ro.far) tok_inputs_load<HPG>(a, ro.g, ro.h, CO ? 0 : 1, in, svr, sgt);
    else tok_inputs_load<HPG>(a, ro.g, ro.g * a.hpg, a.hpg, in, svr, sgt);
    float Mo = -INFINITY;
    o1_ff Zo = ff_make(0.f, 0.f);
    const int b0 = ro.fc * a.MB, nbf = ro.far ? max(0, min(a.MB, a.m - b0)) : 0;
    if (warp == 1 && lane < nbf) {   // the far chunk's entering max and mass (the insert's warp)
        const size_t at = (size_t)ro.h * a.m + b0 + lane;
        Mo = a.M[at];
        Zo = ff_make(a.Z[at], a.Zlo[at]);
    }
    if (tid == 0) {
        const long long p1 = tok_ld_relaxed((const long long *)&a.hdr->pos);
        int mt1[4];
        for (int i = 0; i < 4; ++i) mt1[i] = (int)tok_ld_relaxed_u32(a.meta + ro.g * 4 + i);
        bool same = a.tok_prefetch && p1 == s_pos;
        for (int i = 0; i < 4; ++i) same = same && mt1[i] == s_meta[i];
        int parity = 0;
        if (!same) {
            if (a.tok_prefetch) {
                // copies of a state that has moved since: let them land first
                tok_wait(bar, 0, O1_WAIT_CYCLES_FULL);
                parity = 1;
            }
            s_pos = p1;
            for (int i = 0; i < 4; ++i) s_meta[i] = mt1[i];
            O1Meta mt;
            mt.len0 = mt1[0];
            mt.head0 = mt1[1];
            mt.farl0 = mt1[2];
            mt.wg = mt1[3];
            tok_issue<CO>(a, ro, mt, sm);
        }
        s_parity = parity;
    }
    __syncthreads();
    O1Meta mt;
    mt.len0 = s_meta[0];
    mt.head0 = s_meta[1];
    mt.farl0 = s_meta[2];
    mt.wg = s_meta[3];
    const long long p = s_pos;
    const bool evict = mt.len0 == mt.wg;
    const int farl1 = mt.farl0 + (evict ? 1 : 0);
    if (p != pguess && tid < (a.d >> 1)) tok_cs(a, inv, p, cs, sn);
    float *kpush = nullptr, *vpush = nullptr;
    if (!ro.far) {
        const int ip = tok_near_plan(a, mt, ro.c).ipush;
        if (ip >= 0) {
            kpush = ns.sK + (size_t)ip * a.d;
            vpush = ns.sV + (size_t)ip * a.dv;
        }
    }
    tok_inputs_finish<HPG>(a, ro.g, ro.far ? (CO ? 0 : 1) : a.hpg, cs, sn, in, sq, sk, kpush, vpush);
    tok_cp_wait();
    tok_wait_copies(a, bar, (uint32_t)s_parity);
    __syncthreads();
    if constexpr (CO) {
        if (ro.hl == 0 && ro.fc == 0)   // the group's rotated key, for the commit
            for (int j = tid; j < a.d; j += blockDim.x) a.kcur[(size_t)ro.g * a.d + j] = sk[j];
        tok_far_insert(a, ro, mt, fs, Mo, Zo);
    } else if (ro.far) {
        tok_far_compute(a, ro, mt, fs, Mo, Zo);
    } else {
        tok_near_compute<HPG>(a, ro, mt, ns);
    }

    // ---- arrival: the last CTA for a head merges it; the last of all commits
    __syncthreads();   // every partial and record of this CTA is written
    if (tid == 0) {
        // release: the CTA's partials, records and state writes (ordered
        // before this thread by the barrier) before its counts; a merger or
        // the committer takes the matching acquire after its count
        asm volatile("fence.acq_rel.gpu;" ::: "memory");
        const unsigned total = (unsigned)(a.NC + a.NF);
        unsigned r[HPG];
        const int nt = CO ? 0 : (ro.far ? 1 : a.hpg);   // no merges in a commit
        const unsigned base = ro.far ? (unsigned)ro.h : (unsigned)(ro.g * a.hpg);
#pragma unroll
        for (int i = 0; i < HPG; ++i) r[i] = i < nt ? atomicAdd(a.tick + base + i, 1u) : 0u;
        const unsigned ra = atomicAdd(a.tick + a.nh + a.G, 1u);
        unsigned mine = 0;
#pragma unroll
        for (int i = 0; i < HPG; ++i)
            if (i < nt && r[i] == total - 1) mine |= 1u << (ro.far ? ro.hl : i);
        const bool last = ra == gridDim.x - 1;
        if (mine || last) asm volatile("fence.acq_rel.gpu;" ::: "memory");
        for (int hl = 0; hl < a.hpg; ++hl)
            if (mine & (1u << hl)) a.tick[ro.g * a.hpg + hl] = 0u;   // every arrival for it is in
        s_mine = mine;
        s_last = last;
    }
    __syncthreads();
    // the commit (last of all) on warp 7, beside the merge on the other
    // warps; the merge reuses the shared memory the CTA's work is done with
    const unsigned mine = s_mine;
    const bool last = s_last;
    if (last && warp == 7) {
        tok_commit_warp(a, p, (int *)(smg + 8 * a.hpg));
    } else if (mine) {
        float *stage = ro.far ? fs.sqt : ns.sK;
        tok_merge<HPG>(a, ro.g, mine, farl1, sgt, smg, stage, (size_t)(smg - stage), s_mbar, last ? 224 : 256);
    }
}

// One instance of the kernel per power of two of heads per group (the
// smallest at least hpg), so that nothing is unrolled to the largest count;
// commits (no near slices, no merges) run the one-head instance of CO.
template <int HPG, bool CO>
static cudaError_t tok_launch(const O1Args &a, cudaStream_t st) {
    static unsigned long long done = 0;
    static size_t dyn_max = 0;   // the kernel's static shared memory taken off the 227 KB a block may hold
    unsigned long long bit = 0;
    if (o1_attrs_needed(&done, &bit)) {
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, k_tok<HPG, CO>);
        if (e != cudaSuccess) return e;
        const size_t dmax = 227 * 1024 - fa.sharedSizeBytes;
        e = cudaFuncSetAttribute(k_tok<HPG, CO>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dmax);
        if (e != cudaSuccess) return e;
        __atomic_store_n(&dyn_max, dmax, __ATOMIC_RELAXED);
        o1_attrs_done(&done, bit);
    }
    if (a.tok_smem > __atomic_load_n(&dyn_max, __ATOMIC_RELAXED)) return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.nh * a.NF + (CO ? 0 : a.G * a.NC), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.dynamicSmemBytes = a.tok_smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaLaunchKernelEx(&cfg, k_tok<HPG, CO>, a);
    return cudaGetLastError();
}

cudaError_t o1_launch_token(const O1Args &a, cudaStream_t st) {
    if (a.tok_commit_only) return tok_launch<1, true>(a, st);
    if (a.hpg <= 1) return tok_launch<1, false>(a, st);
    if (a.hpg <= 2) return tok_launch<2, false>(a, st);
    if (a.hpg <= 4) return tok_launch<4, false>(a, st);
    if (a.hpg <= 8) return tok_launch<8, false>(a, st);
    return tok_launch<16, false>(a, st);
}
