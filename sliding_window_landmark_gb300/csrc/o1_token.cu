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
//      row's own rotated key, so the ring is not written before every block
//      has read it), scores for every head of the group, a slice-local
//      softmax -> partial (max, sum, value sum) per head.
//    far blocks (one per head): the evicted key's far insert (M, Z, T in
//      place) fused with the far readout, which reads the updated T once.
//  k_tok_merge  launched with programmatic dependent launch: waits for the
//      main grid, merges the slices and the far part under one exponent
//      (1e-30 floor), gates, and one block commits ring slot, meta and
//      position.
// Nothing waits on a flag: the only dependency is the launch order.
#include <math.h>

#include "o1_common.cuh"

__device__ __forceinline__ void o1_allow_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }
__device__ __forceinline__ void o1_wait_primary() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

static size_t tok_main_smem(const O1Args &a) {
    const size_t near = (size_t)a.hpg * a.d + a.d + (size_t)a.KC * (a.d + a.dv) + (size_t)a.KC * a.hpg + 2 * a.hpg;
    const size_t far = 2 * (size_t)a.d + a.dv + 7 * (size_t)a.m + 32;
    return 4 * (near > far ? near : far);
}

__device__ void tok_near(const O1Args &a, int g, int c, const O1Meta &mt, float *sm) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int d = a.d, dv = a.dv, hpg = a.hpg, half = d >> 1;
    const bool evict = mt.len0 == mt.wg;
    const int len1 = evict ? mt.wg : mt.len0 + 1;
    const int head1 = evict ? (mt.head0 + 1) % mt.wg : mt.head0;
    const int pslot = (mt.head0 + mt.len0) % mt.wg;
    const int n = a.ns + len1;
    const int i0 = c * a.KC;
    const int cnt = max(0, min(a.KC, n - i0));
    float *part = a.part + (size_t)(g * a.NC + c) * hpg * (2 + dv);
    const long long p = a.hdr->pos;

    float *sq = sm;                    // [hpg][d]
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
    // rotate the group's queries and its key
    for (int j = tid; j < half; j += blockDim.x) {
        float cs = 1.f, sn = 0.f;
        if (a.rotate) o1_rope_cs(a.hdr->inv_freq[j], p, cs, sn);
        for (int h = 0; h < hpg; ++h) {
            const float *x = a.q + (size_t)(g * hpg + h) * d;
            const float x0 = x[j], x1 = x[j + half];
            sq[h * d + j] = x0 * cs - x1 * sn;
            sq[h * d + j + half] = x1 * cs + x0 * sn;
        }
        const float *x = a.k + (size_t)g * d;
        const float x0 = x[j], x1 = x[j + half];
        sk[j] = x0 * cs - x1 * sn;
        sk[j + half] = x1 * cs + x0 * sn;
    }
    // the slice's keys and values (the pushed slot's key comes from sk below)
    const int d4 = d >> 2, dv4 = dv >> 2;
    for (int idx = tid; idx < cnt * d4; idx += blockDim.x) {
        const int i = idx / d4, c4 = idx % d4, key = i0 + i;
        const float *src = nullptr;
        if (key < a.ns) src = a.sink_k + ((size_t)g * a.ns + key) * d;
        else {
            const int slot = (head1 + key - a.ns) % mt.wg;
            if (slot != pslot) src = a.ring_k + ((size_t)g * a.w + slot) * d;
        }
        if (src) ((float4 *)(sK + i * d))[c4] = ((const float4 *)src)[c4];
    }
    for (int idx = tid; idx < cnt * dv4; idx += blockDim.x) {
        const int i = idx / dv4, c4 = idx % dv4, key = i0 + i;
        const float *src;
        if (key < a.ns) src = a.sink_v + ((size_t)g * a.ns + key) * dv;
        else {
            const int slot = (head1 + key - a.ns) % mt.wg;
            src = slot == pslot ? a.v + (size_t)g * dv : a.ring_v + ((size_t)g * a.w + slot) * dv;
        }
        ((float4 *)(sV + i * dv))[c4] = ((const float4 *)src)[c4];
    }
    __syncthreads();
    if (c == 0)
        for (int j = tid; j < d; j += blockDim.x) a.kcur[(size_t)g * d + j] = sk[j];
    for (int i = 0; i < cnt; ++i) {
        const int key = i0 + i;
        if (key >= a.ns && (head1 + key - a.ns) % mt.wg == pslot)
            for (int j = tid; j < d; j += blockDim.x) sK[i * d + j] = sk[j];
    }
    if (cnt == 0) return;   // slice 0 of an empty set only publishes the key
    __syncthreads();
    // scores: one warp per (key, head) pair, lanes across d
    for (int pr = warp; pr < cnt * hpg; pr += blockDim.x >> 5) {
        const int i = pr / hpg, h = pr % hpg;
        float s = 0.f;
        for (int j = lane; j < d; j += 32) s = fmaf(sq[h * d + j], sK[i * d + j], s);
        s = warp_sum(s);
        if (lane == 0) sS[i * hpg + h] = s * a.scale;
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
    for (int idx = tid; idx < hpg * dv; idx += blockDim.x) {
        const int h = idx / dv, t = idx % dv;
        float acc = 0.f;
        for (int i = 0; i < cnt; ++i) acc = fmaf(sS[i * hpg + h], sV[i * dv + t], acc);
        part[h * (2 + dv) + 2 + t] = acc;
    }
    for (int h = tid; h < hpg; h += blockDim.x) {
        part[h * (2 + dv)] = sML[2 * h];
        part[h * (2 + dv) + 1] = sML[2 * h + 1];
    }
}

__device__ void tok_far(const O1Args &a, int g, int hl, const O1Meta &mt, float *sm) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
    const int d = a.d, dv = a.dv, m = a.m, half = d >> 1;
    const int h = g * a.hpg + hl;
    const bool evict = mt.len0 == mt.wg;
    const int farl1 = mt.farl0 + (evict ? 1 : 0);
    float *fp = a.farp + (size_t)h * (4 + dv);
    if (farl1 == 0) {
        for (int idx = tid; idx < 4 + dv; idx += blockDim.x) fp[idx] = idx == 0 ? -INFINITY : 0.f;
        return;
    }
    float *sq = sm;             // [d]
    float *ske = sq + d;        // [d]
    float *sve = ske + d;       // [dv]
    float *sMn = sve + dv;      // [m] far max after the insert
    float *sZn = sMn + m;       // [m] far mass after the insert
    float *sRho = sZn + m;      // [m]
    float *sE = sRho + m;       // [m]
    float *sF = sE + m;         // [m] landmark scores, then e^{f - F}
    float *sG = sF + m;         // [m] u, then gains
    float *sC = sG + m;         // [m] F + M_b
    float *sRed = sC + m;       // [32]
    const long long p = a.hdr->pos;
    for (int j = tid; j < half; j += blockDim.x) {
        float cs = 1.f, sn = 0.f;
        if (a.rotate) o1_rope_cs(a.hdr->inv_freq[j], p, cs, sn);
        const float *x = a.q + (size_t)h * d;
        const float x0 = x[j], x1 = x[j + half];
        sq[j] = x0 * cs - x1 * sn;
        sq[j + half] = x1 * cs + x0 * sn;
    }
    if (evict) {
        const float *kk = a.ring_k + ((size_t)g * a.w + mt.head0) * d;
        const float *vv = a.ring_v + ((size_t)g * a.w + mt.head0) * dv;
        for (int j = tid; j < d; j += blockDim.x) ske[j] = kk[j];
        for (int j = tid; j < dv; j += blockDim.x) sve[j] = vv[j];
    }
    __syncthreads();
    // far insert of the evicted key (o1b_far_e / o1b_far_commit for one row)
    if (evict) {
        for (int b = warp; b < m; b += nw) {
            const float *qt = a.qt + ((size_t)h * m + b) * d;
            float s = 0.f;
            for (int j = lane; j < d; j += 32) s = fmaf(qt[j], ske[j], s);
            s = warp_sum(s);
            if (lane == 0) {
                const float l = s * a.scale;
                const float Mo = a.M[(size_t)h * m + b], Zo = a.Z[(size_t)h * m + b];
                const float Mn = fmaxf(Mo, l);
                const float rho = (Mn == Mo) ? 1.f : expf(Mo - Mn);
                const float e = expf(l - Mn);
                const float Zn = Zo * rho + e;
                a.M[(size_t)h * m + b] = Mn;
                a.Z[(size_t)h * m + b] = Zn;
                sMn[b] = Mn;
                sZn[b] = Zn;
                sRho[b] = rho;
                sE[b] = e;
            }
        }
    } else {
        for (int b = tid; b < m; b += blockDim.x) {
            sMn[b] = a.M[(size_t)h * m + b];
            sZn[b] = a.Z[(size_t)h * m + b];
            sRho[b] = 1.f;
            sE[b] = 0.f;
        }
    }
    // landmark scores
    for (int aa = warp; aa < m; aa += nw) {
        const float *kt = a.kt + ((size_t)g * m + aa) * d;
        float s = 0.f;
        for (int j = lane; j < d; j += 32) s = fmaf(sq[j], kt[j], s);
        s = warp_sum(s);
        if (lane == 0) sF[aa] = s * a.scale;
    }
    __syncthreads();
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
        const float *mu = a.mu + (size_t)h * m * m + b;
        float u = 0.f;
        for (int aa = 0; aa < m; ++aa) u = fmaf(sF[aa], mu[(size_t)aa * m], u);
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
    // value sums: insert the evicted value and read the far numerator
    // (16 loads issued before the first store: the stores may alias later
    // loads as far as the compiler knows, which would serialise them)
    for (int t = tid; t < dv; t += blockDim.x) {
        float *T = a.T + (size_t)h * m * dv + t;
        const float vt = evict ? sve[t] : 0.f;
        float acc = 0.f;
        for (int b0 = 0; b0 < m; b0 += 16) {
            float Tv[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) Tv[i] = b0 + i < m ? T[(size_t)(b0 + i) * dv] : 0.f;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int b = b0 + i;
                if (b < m) {
                    float x = Tv[i];
                    if (evict) {
                        x = sRho[b] * x + sE[b] * vt;
                        T[(size_t)b * dv] = x;
                    }
                    acc = fmaf(sG[b], x, acc);
                }
            }
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
    extern __shared__ float sm[];
    o1_allow_dependents();
    const int per = a.NC + a.hpg;
    const int g = blockIdx.x / per, r = blockIdx.x % per;
    const O1Meta mt = o1_meta(a, g);
    if (r < a.NC) tok_near(a, g, r, mt, sm);
    else tok_far(a, g, r - a.NC, mt, sm);
}

// Merge per (head, 64 value columns), 256 threads: the slices' common max
// and mass by block reductions, then four slice groups of 64 columns each
// accumulate with independent loads; block (0, 0) also commits the row.
__global__ __launch_bounds__(256) void k_tok_merge(O1Args a) {
    __shared__ float sred[8];
    __shared__ float sacc[4][64];
    o1_wait_primary();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int h = blockIdx.x, g = h / a.hpg, hl = h % a.hpg;
    const size_t cs = (size_t)a.hpg * (2 + a.dv);
    const float *part = a.part + (size_t)g * a.NC * cs + (size_t)hl * (2 + a.dv);
    float mx = -INFINITY;
    for (int c = tid; c < a.NC; c += 256) mx = fmaxf(mx, __ldcg(part + c * cs));
    mx = warp_max(mx);
    if (lane == 0) sred[warp] = mx;
    __syncthreads();
    mx = sred[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) mx = fmaxf(mx, sred[i]);
    __syncthreads();
    float l = 0.f;
    for (int c = tid; c < a.NC; c += 256) {
        const float mc = __ldcg(part + c * cs);
        if (mc > -INFINITY) l = fmaf(expf(mc - mx), __ldcg(part + c * cs + 1), l);
    }
    l = warp_sum(l);
    if (lane == 0) sred[warp] = l;
    __syncthreads();
    l = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) l += sred[i];
    const int cg = tid >> 6, col = tid & 63, t = blockIdx.y * 64 + col;
    float acc = 0.f;
    if (t < a.dv) {
        float ac[4] = {0.f, 0.f, 0.f, 0.f};
        for (int c0 = cg; c0 < a.NC; c0 += 16) {
            float mc[4], vc[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int c = c0 + 4 * u;
                mc[u] = c < a.NC ? __ldcg(part + c * cs) : -INFINITY;
                vc[u] = c < a.NC ? __ldcg(part + c * cs + 2 + t) : 0.f;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (mc[u] > -INFINITY) ac[u] = fmaf(expf(mc[u] - mx), vc[u], ac[u]);
        }
        acc = (ac[0] + ac[1]) + (ac[2] + ac[3]);
    }
    sacc[cg][col] = acc;
    __syncthreads();
    if (cg == 0 && t < a.dv) {
        acc = (sacc[0][col] + sacc[1][col]) + (sacc[2][col] + sacc[3][col]);
        const float *fp = a.farp + (size_t)h * (4 + a.dv);
        const float cf = __ldcg(fp), Df = __ldcg(fp + 1);
        const bool have = __ldcg(fp + 2) > 0.5f;
        const float c = cf > -INFINITY ? fmaxf(mx, cf) : mx;
        const float al = expf(mx - c);
        const float be = have ? expf(cf - c) : 0.f;
        const float den = fmaxf(be * Df + al * l, 1e-30f);
        float y = (be * __ldcg(fp + 4 + t) + al * acc) / den;
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
