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
    s.smg = s.sP + (size_t)8 * a.KC * a.hpg;
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
    s.smg = (float *)(((uintptr_t)(s.sNum + 256) + 15) & ~(uintptr_t)15);   // 16-byte aligned
    return s;
}

// Thread 0: the copies of the state a CTA needs, for meta `mt`.
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

// A near slice: scores of every head of the group over the slice's keys, a
// slice-local softmax and the value sums -> partial (max, sum, value sum).
template <int HPG>
__device__ void tok_near_compute(const O1Args &a, const TokRole &ro, const O1Meta &mt, const TokNearSm &s) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int d = a.d, dv = a.dv, hpg = a.hpg, KC = a.KC;
    const TokNear p = tok_near_plan(a, mt, ro.c);
    const int cnt = p.cnt;
    const size_t slot = (size_t)(ro.g * a.NC + ro.c) * hpg;
    float *pv = a.part + slot * dv;   // [hpg][dv]
    float *pml = a.pml + slot * 2;    // [hpg][2]
    if (ro.c == 0)   // the group's rotated key, for the commit
        for (int j = tid; j < d; j += blockDim.x) a.kcur[(size_t)ro.g * d + j] = s.sk[j];
    if (cnt == 0) {
        for (int h = tid; h < hpg; h += blockDim.x) {
            pml[2 * h] = -INFINITY;
            pml[2 * h + 1] = 0.f;
        }
        return;
    }
    // (the pushed key's row holds the row's own rotated key and value)
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
#pragma unroll 4
        for (int i = 0; i < cnt; ++i) {
            const float w = s.sS[i * hpg + h];
            const float4 v = ((const float4 *)(s.sV + (size_t)i * dv))[c4];
            acc.x = fmaf(w, v.x, acc.x);
            acc.y = fmaf(w, v.y, acc.y);
            acc.z = fmaf(w, v.z, acc.z);
            acc.w = fmaf(w, v.w, acc.w);
        }
        ((float4 *)(pv + (size_t)h * dv))[c4] = acc;
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
    for (int a0 = 0; a0 < m; a0 += 32) {
        const int aa = a0 + lane;
        float f1[1];
        tok_dots(s.skt, aa, aa < m, s.sq, 0, 1, d, f1);
        if (aa < m) s.sPf[warp * m + aa] = f1[0];
    }
    {
        float l1[1];
        tok_dots(s.sqt, lane, evict && lane < nb, s.ske, 0, 1, d, l1);
        if (lane < nb) s.sPl[warp * MB + lane] = l1[0];
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

// The merge of the heads in `mine` (bits hl of group g), by the CTA that
// arrived last for them: per head, the near slices' (max, sum) -> the window
// max M_w and mass L; the far records -> c_f and D (float-float, sign decision);
// then per (head, 4 columns) the slices' value sums (each moved to M_w), the
// far numerator, one exponent c = max(M_w, c_f) (the far max counts even
// when the far part is dropped, as the pages' c_all does), the 1e-30 floor
// and the gate. The value sums are read as float4, a thread's 16 slices in
// flight at once, the threads split over slice groups when there are more
// threads than (head, 4 columns); nothing in shared memory grows with the
// number of slices.
template <int HPG>
__device__ void tok_merge(const O1Args &a, int g, unsigned mine, int farl1, const float *sgt, float *smg) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int hpg = a.hpg, NC = a.NC, NF = a.NF, dv = a.dv, dv4 = dv >> 2;
    int heads[HPG];
    int nS = 0;
    for (int hl = 0; hl < hpg; ++hl)
        if (mine & (1u << hl)) heads[nS++] = hl;
    float *shd = smg;                       // [nS][8]  M_w, L, c_f, have, D
    float *sff = shd + 8 * nS;              // [nS][NF] far record factors e^{c_r - c_f}
    float4 *sacc = (float4 *)(((uintptr_t)(smg + (size_t)hpg * (NF + 8)) + 15) & ~(uintptr_t)15);   // [256]
    const float *pml = a.pml + (size_t)g * NC * hpg * 2;   // slice c, head hl: pml[(c hpg + hl) 2]
    for (int si = warp; si < nS; si += blockDim.x >> 5) {
        const int hl = heads[si];
        const int h = g * hpg + hl;
        // the far records (c_r, -, D high, D low) and the slices' (max, sum),
        // every load of the lane issued before any is used: NF <= 64, and a
        // lane takes the slices lane, lane + 32, ... with an online max
        float4 fr4[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int r = lane + 32 * k;
            fr4[k] = r < NF ? __ldcg((const float4 *)(a.farp + ((size_t)h * NF + r) * (4 + dv)))
                            : make_float4(-INFINITY, 0.f, 0.f, 0.f);
        }
        float mx = -INFINITY, L = 0.f;
        for (int c = lane; c < NC; c += 32) {
            const float2 v = __ldcg((const float2 *)(pml + ((size_t)c * hpg + hl) * 2));
            if (v.x == -INFINITY) continue;
            const float mn = fmaxf(mx, v.x);
            L = L * expf(mx - mn) + v.y * expf(v.x - mn);
            mx = mn;
        }
        const float Mw = warp_max(mx);
        L = warp_sum(mx == -INFINITY ? 0.f : L * expf(mx - Mw));
        const float cf = warp_max(fmaxf(fr4[0].x, fr4[1].x));
        o1_ff D = ff_make(0.f, 0.f);
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int r = lane + 32 * k;
            const float fr = (fr4[k].x == -INFINITY) ? 0.f : expf(fr4[k].x - cf);
            if (r < NF) sff[si * NF + r] = fr;
            D = ff_add(D, ff_mul_f(ff_make(fr4[k].z, fr4[k].w), fr));
        }
        D = warp_sum(D);
        const float mx_ = Mw;
        if (lane == 0) {
            const bool have = farl1 > 0 && ff_nonneg(D);
            shd[si * 8 + 0] = mx_;
            shd[si * 8 + 1] = L;
            shd[si * 8 + 2] = farl1 > 0 ? cf : -INFINITY;
            shd[si * 8 + 3] = have ? 1.f : 0.f;
            shd[si * 8 + 4] = have ? D.hi + D.lo : 0.f;
        }
    }
    __syncthreads();
    const int items = nS * dv4;
    int nsg = items >= (int)blockDim.x ? 1 : (int)blockDim.x / items;
    if (nsg > 8) nsg = 8;
    for (int it0 = 0; it0 < items; it0 += blockDim.x / nsg) {
        const int it = it0 + tid % (blockDim.x / nsg), sg = tid / (blockDim.x / nsg);
        const bool act = it < items && sg < nsg;
        float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
        int si = 0, c4 = 0;
        if (act) {
            si = it / dv4;
            c4 = it - si * dv4;
            const int hl = heads[si];
            const float Mw = shd[si * 8 + 0];
            const float4 *pv = (const float4 *)(a.part + ((size_t)g * NC * hpg + hl) * dv) + c4;   // slice c: + c hpg dv4
            for (int c0 = sg; c0 < NC; c0 += 16 * nsg) {
                float4 v[16];
                float mc[16];
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const int c = c0 + u * nsg;
                    const bool in = c < NC;
                    mc[u] = in ? __ldcg(pml + ((size_t)c * hpg + hl) * 2) : -INFINITY;
                    v[u] = in ? __ldcg(pv + (size_t)c * hpg * dv4) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    if (mc[u] == -INFINITY) continue;
                    const float f = expf(mc[u] - Mw);
                    A.x = fmaf(f, v[u].x, A.x);
                    A.y = fmaf(f, v[u].y, A.y);
                    A.z = fmaf(f, v[u].z, A.z);
                    A.w = fmaf(f, v[u].w, A.w);
                }
            }
        }
        if (nsg > 1) {
            sacc[tid] = A;
            __syncthreads();
            if (act && sg == 0)
                for (int q = 1; q < nsg; ++q) {
                    const float4 o = sacc[q * (blockDim.x / nsg) + tid];
                    A.x += o.x;
                    A.y += o.y;
                    A.z += o.z;
                    A.w += o.w;
                }
            __syncthreads();
        }
        if (act && sg == 0) {
            const int hl = heads[si], h = g * hpg + hl;
            float4 FN = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int r = 0; r < NF; ++r) {
                const float fr = sff[si * NF + r];
                const float4 n = __ldcg((const float4 *)(a.farp + ((size_t)h * NF + r) * (4 + dv) + 4) + c4);
                FN.x = fmaf(fr, n.x, FN.x);
                FN.y = fmaf(fr, n.y, FN.y);
                FN.z = fmaf(fr, n.z, FN.z);
                FN.w = fmaf(fr, n.w, FN.w);
            }
            const float Mw = shd[si * 8 + 0], L = shd[si * 8 + 1], cf = shd[si * 8 + 2];
            const bool have = shd[si * 8 + 3] > 0.5f;
            const float c = cf > -INFINITY ? fmaxf(Mw, cf) : Mw;
            const float al = expf(Mw - c);
            const float be = have ? expf(cf - c) : 0.f;
            const float rden = 1.f / fmaxf(be * shd[si * 8 + 4] + al * L, 1e-30f);
            float y[4] = {(be * FN.x + al * A.x) * rden, (be * FN.y + al * A.y) * rden, (be * FN.z + al * A.z) * rden,
                          (be * FN.w + al * A.w) * rden};
            if (a.gate)
#pragma unroll
                for (int j = 0; j < 4; ++j) y[j] = y[j] / (1.f + expf(-sgt[hl * dv + 4 * c4 + j]));
            *((float4 *)(a.out + (size_t)h * dv) + c4) = make_float4(y[0], y[1], y[2], y[3]);
        }
    }
}

// The commit of the step, by the CTA that arrived last of all (every CTA has
// read the ring, meta and far state by then): each group's ring slot gets
// the row's rotated key and value and its meta moves (o1b_ring_commit /
// o1b_meta for one row); then the position, the step's last write, released
// after every state write of the step.
__device__ void tok_commit(const O1Args &a, long long p, float *smg) {
    const int tid = threadIdx.x;
    int *sslot = (int *)smg;   // [G] the slot each group pushes to
    for (int g = tid; g < a.G; g += blockDim.x) {
        const int len0 = (int)tok_ld_relaxed_u32(a.meta + g * 4 + 0), head0 = (int)tok_ld_relaxed_u32(a.meta + g * 4 + 1);
        const int farl0 = (int)tok_ld_relaxed_u32(a.meta + g * 4 + 2), wg = (int)tok_ld_relaxed_u32(a.meta + g * 4 + 3);
        sslot[g] = (head0 + len0) % wg;
        if (len0 == wg) {
            a.meta[g * 4 + 1] = (uint32_t)((head0 + 1) % wg);
            a.meta[g * 4 + 2] = (uint32_t)(farl0 + 1);
        } else {
            a.meta[g * 4 + 0] = (uint32_t)(len0 + 1);
        }
    }
    __syncthreads();
    for (size_t i = tid; i < (size_t)a.G * a.d; i += blockDim.x) {
        const int g = (int)(i / a.d), j = (int)(i - (size_t)g * a.d);
        a.ring_k[((size_t)g * a.w + sslot[g]) * a.d + j] = __ldcg(a.kcur + i);
    }
    for (size_t i = tid; i < (size_t)a.G * a.dv; i += blockDim.x) {
        const int g = (int)(i / a.dv), j = (int)(i - (size_t)g * a.dv);
        a.ring_v[((size_t)g * a.w + sslot[g]) * a.dv + j] = a.v[i];
    }
    __syncthreads();
    if (tid == 0) {
        a.tick[a.nh + a.G] = 0u;
        __threadfence();
        tok_st_release((long long *)&a.hdr->pos, p + 1);
    }
}

}  // namespace

template <int HPG>
__global__ __launch_bounds__(256) void k_tok(O1Args a) {
    extern __shared__ __align__(16) float sm[];
    __shared__ long long s_pos;
    __shared__ int s_meta[4];
    __shared__ int s_parity;
    __shared__ unsigned s_mine;
    __shared__ int s_last;
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
            tok_issue(a, ro, mt, sm);
        }
    }
    const float inv = tid < (a.d >> 1) ? a.hdr->inv_freq[tid] : 0.f;   // a constant of the layer
    if (ro.far) {   // mu's columns of the chunk: a constant of the layer
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
    if (ro.far) tok_inputs_load<HPG>(a, ro.g, ro.h, 1, in, svr, sgt);
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
            tok_issue(a, ro, mt, sm);
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
    tok_inputs_finish<HPG>(a, ro.g, ro.far ? 1 : a.hpg, cs, sn, in, sq, sk, kpush, vpush);
    tok_cp_wait();
    tok_wait_copies(a, bar, (uint32_t)s_parity);
    __syncthreads();
    if (ro.far) tok_far_compute(a, ro, mt, fs, Mo, Zo);
    else tok_near_compute<HPG>(a, ro, mt, ns);

    // ---- arrival: the last CTA for a head merges it; the last of all commits
    __syncthreads();   // every partial and record of this CTA is written
    if (tid == 0) {
        __threadfence();
        const unsigned total = (unsigned)(a.NC + a.NF);
        unsigned r[HPG];
        const int nt = ro.far ? 1 : a.hpg;
        const unsigned base = ro.far ? (unsigned)ro.h : (unsigned)(ro.g * a.hpg);
#pragma unroll
        for (int i = 0; i < HPG; ++i) r[i] = i < nt ? atomicAdd(a.tick + base + i, 1u) : 0u;
        const unsigned ra = atomicAdd(a.tick + a.nh + a.G, 1u);
        unsigned mine = 0;
#pragma unroll
        for (int i = 0; i < HPG; ++i)
            if (i < nt && r[i] == total - 1) mine |= 1u << (ro.far ? ro.hl : i);
        const bool last = ra == gridDim.x - 1;
        if (mine || last) __threadfence();
        for (int hl = 0; hl < a.hpg; ++hl)
            if (mine & (1u << hl)) a.tick[ro.g * a.hpg + hl] = 0u;   // every arrival for it is in
        s_mine = mine;
        s_last = last;
    }
    __syncthreads();
    if (s_mine) tok_merge<HPG>(a, ro.g, s_mine, farl1, sgt, smg);
    if (s_last) {
        __syncthreads();
        tok_commit(a, p, smg);
    }
}

// One instance of the kernel per power of two of heads per group (the
// smallest at least hpg), so that nothing is unrolled to the largest count.
template <int HPG>
static cudaError_t tok_launch(const O1Args &a, cudaStream_t st) {
    static unsigned long long done = 0;
    static size_t dyn_max = 0;   // the kernel's static shared memory taken off the 227 KB a block may hold
    unsigned long long bit = 0;
    if (o1_attrs_needed(&done, &bit)) {
        cudaFuncAttributes fa;
        cudaError_t e = cudaFuncGetAttributes(&fa, k_tok<HPG>);
        if (e != cudaSuccess) return e;
        const size_t dmax = 227 * 1024 - fa.sharedSizeBytes;
        e = cudaFuncSetAttribute(k_tok<HPG>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dmax);
        if (e != cudaSuccess) return e;
        __atomic_store_n(&dyn_max, dmax, __ATOMIC_RELAXED);
        o1_attrs_done(&done, bit);
    }
    if (a.tok_smem > __atomic_load_n(&dyn_max, __ATOMIC_RELAXED)) return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.nh * a.NF + a.G * a.NC, 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.dynamicSmemBytes = a.tok_smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaLaunchKernelEx(&cfg, k_tok<HPG>, a);
    return cudaGetLastError();
}

cudaError_t o1_launch_token(const O1Args &a, cudaStream_t st) {
    if (a.hpg <= 1) return tok_launch<1>(a, st);
    if (a.hpg <= 2) return tok_launch<2>(a, st);
    if (a.hpg <= 4) return tok_launch<4>(a, st);
    if (a.hpg <= 8) return tok_launch<8>(a, st);
    return tok_launch<16>(a, st);
}
