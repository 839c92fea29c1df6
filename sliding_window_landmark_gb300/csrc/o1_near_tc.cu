// The sliding-window part of a chunk on the 5th-generation tensor cores
// (tcgen05, TMEM accumulators, TMA-staged operands), with fp32 accuracy from
// fp16 tensor-core passes: every fp32 operand x is split into x_hi = fp16(x)
// and x_lo = fp16(x - x_hi) (22 significant bits together), and each product
// is taken as hi.hi + hi.lo + lo.hi (the dropped lo.lo term is ~2^-22
// relative) — the error-compensated split of Markidis et al. (2018) and
// Ootomo & Yokota (2022), here with fp16 halves and fp32 accumulation. fp16
// passes run at twice the tf32 rate, so the three cost about 1.5 tf32 passes;
// a single tf32 pass misses the 1e-4 tolerance on rows whose window holds
// only a few keys.
//
// The pages run the window as a per-row loop over keys (o1_batch.rs,
// o1b_attend) or, on Metal, as two GEMMs over a gathered panel of window
// keys and values (o1c.rs, attend_gemm: o1c_gather, S = q.kp^T, masked
// softmax, O = S.vp). This is the second shape, fused:
//
//  k_gather_tc  per group, the window key sequence X = [ring, oldest first]
//               ++ [this pass's rotated keys] as dense fp16 panels
//               Xk[hi|lo][g][x][d] and, transposed, XvT[hi|lo][g][t][x],
//               zero past the end.
//  k_near_tc    one CTA per (128 query rows, head): Q_hi and Q_lo resident in
//               smem (128-byte swizzle); key tiles of 128 stream through a
//               TMA ring (a key d-chunk or a value half-tile per 32 KB slot);
//               S = Q.K^T (N = 128) into one of two TMEM buffers; softmax
//               threads (one per row) mask to the row's window, keep a
//               running max, write P (hi and lo, fp16) back over S in TMEM;
//               O += P.V with P read from TMEM. The epilogue writes the
//               window numerator O to `out` through shared memory with
//               coalesced stores, and each row's (reference, mass, true max)
//               to its window header; k_merge (o1_chunk.cu) adds the
//               side part under one exponent and gates.
//
// Tile width: a 128 x N x 16 MMA costs about the same time on the tensor
// pipe for N = 64 and N = 128, so S is issued with N = 128 (48 MMAs per
// 128 keys at d = 256 instead of 96); that needs both S buffers at 128
// columns, so with O at up to 256 columns the TMEM is full and Q_lo stays
// in smem (an SS MMA for lo.hi costs the same as the TS form).
//
// Roles: warps 0-3 softmax / epilogue (thread = TMEM lane = query row),
// warp 4 TMA producer, warp 5 MMA issuer (and TMEM owner). Every wait is
// bounded by a clock limit; on expiry the kernel raises a flag in the state
// header and stops issuing work, then waits (with the full limit) for the
// MMAs and copies it has already issued before it releases its TMEM and
// shared memory.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <math.h>

#include "o1_common.cuh"

namespace {

constexpr int TC_BM = O1_TC_BM;    // query rows per CTA
constexpr int TC_BN = O1_TC_BN;    // keys per tile
constexpr int TC_SLOT = 32768;     // bytes per ring slot
constexpr int TC_THREADS = 192;
constexpr int TC_O_COL = 0;        // O accumulator: TMEM columns [0, dv)
constexpr int TC_S_COL = 256;      // S / P buffers: [256, 384) and [384, 512)
constexpr float TC_RESCALE = 8.f;  // log2-units headroom before O is rescaled

__device__ __forceinline__ uint32_t su32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ bool mbar_try(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(su32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait: false (and the shared abort flag raised) after `limit`
// cycles or once another thread has aborted.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort, long long limit) {
    if (mbar_try(bar, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        if (mbar_try(bar, parity)) return true;
        if (*abort) return false;
        if (clock64() - t0 > limit) {
            *abort = 1;
            return false;
        }
    }
}
// Drain: wait, with the full limit, for a phase whose operations are already
// in flight (copies or MMAs that write this block's shared memory or TMEM).
__device__ __forceinline__ void mbar_drain(uint64_t *bar, uint32_t parity) {
    const long long t0 = clock64();
    while (!mbar_try(bar, parity) && clock64() - t0 < O1_WAIT_CYCLES_FULL) {
    }
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void tma_3d(void *dst, const CUtensorMap *map, int x, int y, int z, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
            su32(dst)),
        "l"((uint64_t)map), "r"(x), "r"(y), "r"(z), "r"(su32(bar))
        : "memory");
}
__device__ __forceinline__ void tma_4d(void *dst, const CUtensorMap *map, int x, int y, int z, int w, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(
            su32(dst)),
        "l"((uint64_t)map), "r"(x), "r"(y), "r"(z), "r"(w), "r"(su32(bar))
        : "memory");
}
__device__ __forceinline__ void tc_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (the layout TMA writes with CU_TENSOR_MAP_SWIZZLE_128B).
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
    uint64_t d = (uint64_t)((saddr & 0x3FFFF) >> 4);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}
// Instruction descriptor, kind::f16: f32 accumulate, f16 A and B, both K-major.
__device__ __forceinline__ uint32_t idesc_f16(int M, int N) {
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\ntcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
        "l"(a), "l"(b), "r"(id), "r"(acc)
        : "memory");
}
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t id, uint32_t acc) {
    asm volatile(
        "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\ntcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d),
        "r"(a), "l"(b), "r"(id), "r"(acc)
        : "memory");
}
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(bar))
                 : "memory");
}
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// (a, b) as fp16 pairs hi = fp16(x), lo = fp16(x - hi) (the subtraction is
// exact), packed with a in the low half
__device__ __forceinline__ void split_pair(float a, float b, uint32_t &hi, uint32_t &lo) {
    const __half2 h = __floats2half2_rn(a, b);
    const float2 hf = __half22float2(h);
    const __half2 l = __floats2half2_rn(a - hf.x, b - hf.y);
    hi = *(const uint32_t *)&h;
    lo = *(const uint32_t *)&l;
}

#define TMEM_LD32(taddr, r)                                                                                          \
    asm volatile(                                                                                                    \
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18," \
        "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"                                               \
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),           \
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),     \
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),   \
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])    \
        : "r"(taddr))
#define TMEM_ST32(taddr, r)                                                                                           \
    asm volatile(                                                                                                     \
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18," \
        "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),                                      \
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), \
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),   \
        "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),   \
        "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])                                                                \
        : "memory")
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// The CTA's tile schedule; every role derives the same one.
struct TcPlan {
    int r0, nr, h, g, kt0, nkc;
    int split, jb, nt;   // key split blockIdx.z: tiles jb .. jb + nt - 1 of the row block
    O1Meta mt;
};

__device__ __forceinline__ TcPlan tc_plan(const O1Args &a) {
    TcPlan p;
    // row blocks in reverse: the late blocks see full windows and are the
    // longest, so they start first and the short early ones fill the tail
    p.r0 = (gridDim.x - 1 - blockIdx.x) * TC_BM;
    p.h = blockIdx.y;
    p.g = p.h / a.hpg;
    p.mt = o1_meta(a, p.g);
    p.nr = min(TC_BM, a.R - p.r0);
    const int lo_first = max(0, p.mt.len0 + p.r0 + 1 - p.mt.wg);
    const int hi_last = p.mt.len0 + p.r0 + p.nr - 1;
    p.kt0 = lo_first & ~7;   // TMA x coordinates of the fp16 value panel: 16-byte aligned
    // a contiguous run of the row block's key tiles per split (gridDim.z
    // splits; a split past the last tile has none and writes an empty header)
    const int ntall = (hi_last - p.kt0) / TC_BN + 1;
    const int per = (ntall + (int)gridDim.z - 1) / (int)gridDim.z;
    p.split = blockIdx.z;
    p.jb = p.split * per;
    p.nt = max(0, min(ntall, p.jb + per) - p.jb);
    p.nkc = a.d / 64;        // 64 fp16 = one 128-byte swizzle row; one ring slot per d-chunk (hi, lo)
    return p;
}

}  // namespace

// ------------------------------------------------------------------ gather

// Block = (32 keys, group). Keys past the sequence are written as zeros so
// that masked columns never meet a non-finite value. Xk holds the hi panel
// [G][NXp][d] then the lo panel; XvT the hi panel [G][dv][NXp] then the lo.
// A value outside the fp16 range raises O1_FLAG_FP16_RANGE in the state
// header's flags.
__global__ __launch_bounds__(256) void k_gather_tc(O1Args a, unsigned short *Xk, unsigned short *XvT, int NXp) {
    __shared__ uint32_t sv[32][O1_MAX_DV / 2 + 1];   // [key][t pair]: hi | lo << 16 per element, two passes
    __shared__ unsigned short svl[32][O1_MAX_DV + 2];
    o1_chain_wait();
    const int g = blockIdx.y, x0 = blockIdx.x * 32;
    const O1Meta mt = o1_meta(a, g);
    const int NX = mt.len0 + a.R;
    const size_t kpanel = (size_t)a.G * NXp * a.d, vpanel = (size_t)a.G * a.dv * NXp;
    bool range_ok = true;
    const int d2 = a.d >> 1;
    // loads in batches of 8 ahead of their stores (the stores could alias
    // later loads as far as the compiler knows, which would serialise them)
    for (int base = threadIdx.x; base < 32 * d2; base += 8 * 256) {
        float2 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int idx = base + 256 * u, i = idx / d2, j2 = idx % d2, x = x0 + i;
            v[u] = (idx < 32 * d2 && x < NX) ? ((const float2 *)o1_key(a, g, x, mt))[j2] : make_float2(0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int idx = base + 256 * u, i = idx / d2, j2 = idx % d2, x = x0 + i;
            if (idx >= 32 * d2 || x >= NXp) continue;
            uint32_t hi, lo;
            split_pair(v[u].x, v[u].y, hi, lo);
            range_ok &= fabsf(v[u].x) < 65504.f && fabsf(v[u].y) < 65504.f;
            const size_t o = ((size_t)g * NXp + x) * a.d + 2 * j2;
            *(uint32_t *)(Xk + o) = hi;
            *(uint32_t *)(Xk + kpanel + o) = lo;
        }
    }
    for (int base = threadIdx.x; base < 32 * a.dv; base += 8 * 256) {
        float v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int idx = base + 256 * u, i = idx / a.dv, t = idx % a.dv, x = x0 + i;
            v[u] = (idx < 32 * a.dv && x < NX) ? o1_val(a, g, x, mt)[t] : 0.f;
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int idx = base + 256 * u, i = idx / a.dv, t = idx % a.dv;
            if (idx >= 32 * a.dv) continue;
            const __half h = __float2half_rn(v[u]);
            const __half l = __float2half_rn(v[u] - __half2float(h));
            range_ok &= fabsf(v[u]) < 65504.f;
            ((unsigned short *)sv[i])[t] = __half_as_ushort(h);
            svl[i][t] = __half_as_ushort(l);
        }
    }
    if (!range_ok) atomicOr(&a.hdr->flags, (uint32_t)O1_FLAG_FP16_RANGE);
    __syncthreads();
    for (int idx = threadIdx.x; idx < 32 * a.dv; idx += blockDim.x) {
        const int t = idx >> 5, i = idx & 31, x = x0 + i;
        if (x < NXp) {
            const size_t o = ((size_t)g * a.dv + t) * NXp + x;
            XvT[o] = ((const unsigned short *)sv[i])[t];
            XvT[vpanel + o] = svl[i][t];
        }
    }
}

// --------------------------------------------------------------- attention

// Shared memory: Q_hi [nkc][128 rows][128 B], Q_lo the same, then nslot ring
// slots of 32 KB, then barriers. A key item is one d-chunk of a 128-key tile
// (hi 16 KB, lo 16 KB); a value item is the hi or lo half of V^T for 64 keys
// (dv rows x 128 B). Per tile j the ring carries K(j) chunks 0..nkc-1, later
// V(j) as hi(keys 0-63), lo(0-63), hi(64-127), lo(64-127).
__global__ __launch_bounds__(TC_THREADS, 1) void k_near_tc(O1Args a, const __grid_constant__ CUtensorMap mk,
                                                            const __grid_constant__ CUtensorMap mv,
                                                            const __grid_constant__ CUtensorMap mq, int NXp, int nslot) {
    extern __shared__ __align__(1024) unsigned char smraw[];
    unsigned char *sm = (unsigned char *)(((uintptr_t)smraw + 1023) & ~(uintptr_t)1023);
    const TcPlan pl = tc_plan(a);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int dv = a.dv;
    unsigned char *sQh = sm;                                 // nkc x 16 KB
    unsigned char *sQl = sQh + (size_t)pl.nkc * 16384;       // nkc x 16 KB
    unsigned char *sR = sQl + (size_t)pl.nkc * 16384;        // nslot x 32 KB
    uint64_t *bars = (uint64_t *)(sR + (size_t)nslot * TC_SLOT);
    uint64_t *full = bars, *empty = bars + nslot;
    uint64_t *s_full = bars + 2 * nslot, *p_full = s_full + 2, *pv_done = p_full + 2, *o_done = pv_done + 1,
             *q_ready = o_done + 1;   // the Q tile's TMA
    uint32_t *tslot = (uint32_t *)(q_ready + 1);
    volatile int *abort = (volatile int *)(tslot + 1);

    if (tid == 0) {
        for (int i = 0; i < nslot; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        mbar_init(&s_full[0], 1);
        mbar_init(&s_full[1], 1);
        mbar_init(&p_full[0], TC_BM);
        mbar_init(&p_full[1], TC_BM);
        mbar_init(pv_done, 1);
        mbar_init(o_done, 1);
        mbar_init(q_ready, 1);
        *abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 5) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tslot)), "r"(512)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_before();
    __syncthreads();
    tc_after();
    // the set-up above overlaps the gather's end; the meta read by tc_plan is
    // written only by the pass's commit, after this kernel
    o1_chain_wait();
    const uint32_t tmem = *tslot;
    const long long wl = a.wait_cycles;   // limit of every wait but the final drains
    int issued = 0;                      // ring items the producer has issued (its lane 0)

    if (warp == 4) {
        // ---------------------------------------------------- TMA producer
        // (starts at once: the Q tile has its own smem)
        if (lane == 0 && pl.nt > 0) {
            // the Q tile, fp16 hi and lo, straight into its swizzled slots
            // (rows past R read as zeros)
            mbar_expect_tx(q_ready, 2 * pl.nkc * 16384);
            for (int hl = 0; hl < 2; ++hl)
                for (int c = 0; c < pl.nkc; ++c)
                    tma_4d((hl ? sQl : sQh) + (size_t)c * 16384, &mq, 64 * c, pl.h, pl.r0, hl, q_ready);
            int it = 0;
            const int ybase = pl.g * NXp;
            auto next = [&](uint32_t bytes) -> int {
                const int s = it % nslot;
                if (!mbar_wait(&empty[s], ((it / nslot) & 1) ^ 1, abort, wl)) return -1;
                mbar_expect_tx(&full[s], bytes);
                ++it;
                return s;
            };
            auto load_k = [&](int j) -> bool {
                for (int c = 0; c < pl.nkc; ++c) {
                    const int s = next(2 * TC_BN * 128);
                    if (s < 0) return false;
                    for (int hl = 0; hl < 2; ++hl)
                        tma_3d(sR + (size_t)s * TC_SLOT + hl * (TC_BN * 128), &mk, 64 * c,
                               ybase + pl.kt0 + TC_BN * (pl.jb + j), hl, &full[s]);
                }
                return true;
            };
            auto load_v = [&](int j) -> bool {
                for (int kh = 0; kh < 2; ++kh)
                    for (int hl = 0; hl < 2; ++hl) {
                        const int s = next(dv * 128);
                        if (s < 0) return false;
                        tma_3d(sR + (size_t)s * TC_SLOT, &mv, pl.kt0 + TC_BN * (pl.jb + j) + 64 * kh, pl.g * dv, hl,
                               &full[s]);
                    }
                return true;
            };
            bool ok = load_k(0);
            for (int j = 0; ok && j < pl.nt; ++j) {
                if (j + 1 < pl.nt) ok = load_k(j + 1);
                if (ok) ok = load_v(j);
            }
            issued = it;   // copies still in flight after an abort are drained at the end
        }
    } else if (warp == 5) {
        // ------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t id_s = idesc_f16(TC_BM, TC_BN), id_o = idesc_f16(TC_BM, dv);
            const uint32_t qh0 = su32(sQh), ql0 = su32(sQl), ra = su32(sR);
            int it = 0;
            bool ok = pl.nt > 0 && mbar_wait(q_ready, 0, abort, wl);
            tc_after();
            // S = Q_hi.K_hi + Q_hi.K_lo + Q_lo.K_hi, one ring slot per d-chunk
            auto issue_s = [&](int j) -> bool {
                const uint32_t dcol = tmem + TC_S_COL + TC_BN * (j & 1);
                for (int c = 0; c < pl.nkc; ++c) {
                    const int s = it % nslot;
                    if (!mbar_wait(&full[s], (it / nslot) & 1, abort, wl)) return false;
                    tc_after();
                    const uint32_t kh = ra + s * TC_SLOT, kl = kh + TC_BN * 128, qh = qh0 + c * 16384,
                                   ql = ql0 + c * 16384;
                    for (int k = 0; k < 4; ++k) {
                        mma_ss(dcol, desc_sw128(qh + 32 * k), desc_sw128(kh + 32 * k), id_s, (c | k) ? 1u : 0u);
                        mma_ss(dcol, desc_sw128(qh + 32 * k), desc_sw128(kl + 32 * k), id_s, 1u);
                        mma_ss(dcol, desc_sw128(ql + 32 * k), desc_sw128(kh + 32 * k), id_s, 1u);
                    }
                    mma_commit(&empty[s]);
                    ++it;
                }
                mma_commit(&s_full[j & 1]);
                return true;
            };
            // O += P_hi.V_hi + P_hi.V_lo + P_lo.V_hi, per 64-key half
            auto issue_pv = [&](int j) -> bool {
                const uint32_t pcol = tmem + TC_S_COL + TC_BN * (j & 1);
                for (int kh = 0; kh < 2; ++kh) {
                    const int sh = it % nslot, sl = (it + 1) % nslot;
                    if (!mbar_wait(&full[sh], (it / nslot) & 1, abort, wl)) return false;
                    if (!mbar_wait(&full[sl], ((it + 1) / nslot) & 1, abort, wl)) return false;
                    tc_after();
                    const uint32_t vh = ra + sh * TC_SLOT, vl = ra + sl * TC_SLOT;
                    for (int k = 0; k < 4; ++k) {
                        const uint32_t ph = pcol + 64 * kh + 16 * k, plo = ph + 8;   // keys 64kh + 16k .. + 15
                        mma_ts(tmem + TC_O_COL, ph, desc_sw128(vh + 32 * k), id_o, (j | kh | k) ? 1u : 0u);
                        mma_ts(tmem + TC_O_COL, ph, desc_sw128(vl + 32 * k), id_o, 1u);
                        mma_ts(tmem + TC_O_COL, plo, desc_sw128(vh + 32 * k), id_o, 1u);
                    }
                    mma_commit(&empty[sh]);
                    mma_commit(&empty[sl]);
                    it += 2;
                }
                mma_commit(pv_done);
                return true;
            };
            if (ok) ok = issue_s(0);
            for (int j = 0; ok && j < pl.nt; ++j) {
                if (j + 1 < pl.nt) ok = issue_s(j + 1);
                if (!ok) break;
                ok = mbar_wait(&p_full[j & 1], (j >> 1) & 1, abort, wl);
                tc_after();
                if (ok) ok = issue_pv(j);
            }
            // o_done is committed even after an abort, so that it tracks every
            // MMA this thread issued before TMEM is released
            mma_commit(o_done);
        }
    } else {
        // ------------------------------------------- softmax and epilogue
        const int row = tid;   // TMEM lane
        const int r = pl.r0 + row;
        const bool valid = row < pl.nr;
        const int lo = max(0, pl.mt.len0 + r + 1 - pl.mt.wg), hi = pl.mt.len0 + r;
        const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
        const float sc2 = a.scale * 1.4426950408889634f;   // scores in log2 units
        float mref = -INFINITY, mtrue = -INFINITY, l = 0.f;
        bool ok = true;
        uint32_t v[64];
        for (int j = 0; j < pl.nt && ok; ++j) {
            ok = __all_sync(0xffffffffu, mbar_wait(&s_full[j & 1], (j >> 1) & 1, abort, wl));
            if (!ok) break;
            tc_after();
            const uint32_t scol = lane_base + TC_S_COL + TC_BN * (j & 1);
            const int x0 = pl.kt0 + TC_BN * (pl.jb + j);
            const bool all_in = valid && x0 >= lo && x0 + TC_BN - 1 <= hi;
            const int a0 = lo - x0, a1 = hi - x0;   // valid columns [a0, a1]
            // pass 1: the tile's row max (scores scaled to log2 units, masked).
            // A tile inside the row's window takes a path without per-column
            // predicates (64 selects on a handful of predicate registers
            // serialise); tiles that cross a window edge take the masked one.
            float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll 1
            for (int hf = 0; hf < 2; ++hf) {
                TMEM_LD32(scol + 64 * hf, (&v[0]));
                TMEM_LD32(scol + 64 * hf + 32, (&v[32]));
                tmem_ld_wait();
                if (all_in) {
#pragma unroll
                    for (int c = 0; c < 64; ++c) m4[c & 3] = fmaxf(m4[c & 3], __uint_as_float(v[c]) * sc2);
                } else {
                    const int b0 = a0 - 64 * hf, b1 = a1 - 64 * hf;   // valid columns of this half
#pragma unroll
                    for (int c = 0; c < 64; ++c) {
                        const bool in = valid && c >= b0 && c <= b1;
                        m4[c & 3] = fmaxf(m4[c & 3], in ? __uint_as_float(v[c]) * sc2 : -INFINITY);
                    }
                }
            }
            const float mt = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
            mtrue = fmaxf(mtrue, mt);
            const bool need = mt > mref + TC_RESCALE;
            if (__any_sync(0xffffffffu, need)) {
                const float mnew = fmaxf(mref, mt);
                if (j > 0) {
                    // O holds PV_0 .. PV_{j-1}: wait for the last of them, then rescale
                    ok = __all_sync(0xffffffffu, mbar_wait(pv_done, (j - 1) & 1, abort, wl));
                    if (!ok) break;
                    tc_after();
                    const float f = mref > -INFINITY ? ex2(mref - mnew) : 0.f;
                    uint32_t o[32];
                    for (int c = 0; c < dv / 32; ++c) {
                        TMEM_LD32(lane_base + TC_O_COL + 32 * c, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int t = 0; t < 32; ++t) o[t] = __float_as_uint(__uint_as_float(o[t]) * f);
                        TMEM_ST32(lane_base + TC_O_COL + 32 * c, o);
                    }
                    tmem_st_wait();
                    l *= f;
                }
                mref = mnew;
            }
            // pass 2: P = 2^(s - mref) as fp16 pairs (two keys per column, the
            // lower key in the low half), per 16-key group q: hi in columns
            // 16q..16q+7, lo in 16q+8..16q+15, written over the scores of the
            // same 64-key half after they are read. No key is valid in this
            // row yet iff mref is -inf.
            const float mr = mref > -INFINITY ? mref : 0.f;
            float ls0 = 0.f, ls1 = 0.f;
#pragma unroll 1
            for (int hf = 0; hf < 2; ++hf) {
                TMEM_LD32(scol + 64 * hf, (&v[0]));
                TMEM_LD32(scol + 64 * hf + 32, (&v[32]));
                tmem_ld_wait();
                // exponent arguments s - mref in place; masked columns -inf
                // (2^-inf = 0), with predicates only on tiles that cross an edge
                if (all_in) {
#pragma unroll
                    for (int c = 0; c < 64; ++c) v[c] = __float_as_uint(fmaf(__uint_as_float(v[c]), sc2, -mr));
                } else {
                    const int b0 = a0 - 64 * hf, b1 = a1 - 64 * hf;
#pragma unroll
                    for (int c = 0; c < 64; ++c) {
                        const bool in = valid && c >= b0 && c <= b1;
                        v[c] = __float_as_uint(in ? fmaf(__uint_as_float(v[c]), sc2, -mr) : -INFINITY);
                    }
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float pq[16];
#pragma unroll
                    for (int t = 0; t < 16; ++t) pq[t] = ex2(__uint_as_float(v[16 * q + t]));
#pragma unroll
                    for (int t = 0; t < 8; ++t) {
                        uint32_t hw, lw;
                        split_pair(pq[2 * t], pq[2 * t + 1], hw, lw);
                        ls0 += pq[2 * t];
                        ls1 += pq[2 * t + 1];
                        v[16 * q + t] = hw;
                        v[16 * q + 8 + t] = lw;
                    }
                }
                TMEM_ST32(scol + 64 * hf, (&v[0]));
                TMEM_ST32(scol + 64 * hf + 32, (&v[32]));
            }
            l += ls0 + ls1;
            tmem_st_wait();
            tc_before();
            mbar_arrive(&p_full[j & 1]);
        }
        ok = __all_sync(0xffffffffu, ok && mbar_wait(o_done, 0, abort, wl));
        tc_after();
        if (ok) {
            // the window part of each row: its header (reference, mass, true
            // max, natural units) and its numerator O, which goes to `out`
            // through shared memory with coalesced stores; the side readout
            // merges it with the sinks and the far field and applies the gate
            // (split s > 0 writes the same into its partial, the merge adds
            // the splits up; a split without tiles writes an empty header)
            const size_t RN = (size_t)a.R * a.nh;
            float *hdr = pl.split == 0 ? a.fh : a.wpart + (size_t)(gridDim.z - 1) * RN * dv + (pl.split - 1) * RN * 4;
            if (valid)
                *(float4 *)(hdr + ((size_t)r * a.nh + pl.h) * 4) = make_float4(
                    mref * 0.6931471805599453f, l, mtrue * 0.6931471805599453f, 0.f);
        }
        if (ok && pl.nt > 0) {
            float *onum = pl.split == 0 ? a.out : a.wpart + (pl.split - 1) * (size_t)a.R * a.nh * dv;
            float *so = (float *)sm;   // Q and the ring are free: every MMA has completed
            const int ostride = dv + 4;
            uint32_t o[32];
            for (int c = 0; c < dv / 32; ++c) {
                TMEM_LD32(lane_base + TC_O_COL + 32 * c, o);
                tmem_ld_wait();
#pragma unroll
                for (int t4 = 0; t4 < 8; ++t4)
                    *(float4 *)(so + row * ostride + 32 * c + 4 * t4) =
                        make_float4(__uint_as_float(o[4 * t4]), __uint_as_float(o[4 * t4 + 1]),
                                    __uint_as_float(o[4 * t4 + 2]), __uint_as_float(o[4 * t4 + 3]));
            }
            asm volatile("bar.sync 1, 128;" ::: "memory");
            const int dv4 = dv >> 2;
            const int n4 = pl.nr * dv4;
            for (int idx = tid; idx < n4; idx += TC_BM) {
                const int i = idx / dv4, c4 = idx % dv4;
                *(float4 *)(onum + ((size_t)(pl.r0 + i) * a.nh + pl.h) * dv + 4 * c4) =
                    *(const float4 *)(so + i * ostride + 4 * c4);
            }
        }
    }
    // everyone waits for the MMA thread's final commit before TMEM is released
    if (warp == 5 && lane == 0) mbar_drain(o_done, 0);
    tc_before();
    __syncthreads();
    tc_after();
    // After an abort (every role has stopped by now, so the flag no longer
    // changes): the producer waits, with the full limit, for its copies that
    // may still be in flight (the Q tile and the last nslot ring items) before
    // the block's shared memory is given up.
    if (warp == 4 && lane == 0 && *abort) {
        if (pl.nt > 0) mbar_drain(q_ready, 0);
        for (int i = max(0, issued - nslot); i < issued; ++i) mbar_drain(&full[i % nslot], (i / nslot) & 1);
    }
    __syncthreads();
    if (warp == 5) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512) : "memory");
    if (tid == 0 && *abort) atomicOr(&a.hdr->flags, (uint32_t)O1_FLAG_WAIT_EXPIRED);
}

// ----------------------------------------------------------------- launch

namespace {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        cudaDriverEntryPointQueryResult q;
        void *p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
    }
    return fn;
}

// A [2][outer][inner] fp16 panel pair (hi, lo), boxes of box_inner x box_outer.
bool make_map(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer, uint32_t box_inner,
              uint32_t box_outer) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {inner, outer, 2};
    cuuint64_t strides[2] = {inner * 2, inner * outer * 2};
    cuuint32_t box[3] = {box_inner, box_outer, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, (void *)base, dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t tc_smem(int d, int *nslot) {
    // alignment slack, Q_hi and Q_lo, barriers + row factors
    const size_t fixed = 1024 + 2 * (size_t)(d / 64) * 16384 + 2048;
    const size_t limit = 227 * 1024;
    int ns = (int)((limit - fixed) / TC_SLOT);
    if (ns > 8) ns = 8;
    *nslot = ns;
    return fixed + (size_t)ns * TC_SLOT;
}

}  // namespace

cudaError_t o1_launch_gather_tc(const O1Args &a, cudaStream_t st) {
    o1_launch_chained(a.chain_early, k_gather_tc, dim3((a.nxp + 31) / 32, a.G), dim3(256), 0, st, a, a.Xk, a.XvT, a.nxp);
    return cudaGetLastError();
}

cudaError_t o1_launch_near_tc(const O1Args &a, cudaStream_t st) {
    static unsigned long long done = 0;
    int nslot = 0;
    const size_t smem = tc_smem(a.d, &nslot);
    const int NXp = a.nxp;
    unsigned long long bit = 0;
    if (o1_attrs_needed(&done, &bit)) {
        cudaFuncSetAttribute(k_near_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
        o1_attrs_done(&done, bit);
    }
    CUtensorMap mk, mv;
    if (!make_map(&mk, a.Xk, (uint64_t)a.d, (uint64_t)a.G * NXp, 64, TC_BN)) return cudaErrorInvalidValue;
    if (!make_map(&mv, a.XvT, (uint64_t)NXp, (uint64_t)a.G * a.dv, 64, (uint32_t)a.dv)) return cudaErrorInvalidValue;
    if (nslot < 3) return cudaErrorInvalidValue;   // a value half-tile needs two slots, plus one in flight
    CUtensorMap mq;
    {
        // Qs [2][R][nh][d] fp16, boxes of 64 x 1 head x 128 rows
        auto enc = tensor_map_encoder();
        if (!enc) return cudaErrorInvalidValue;
        cuuint64_t dims[4] = {(cuuint64_t)a.d, (cuuint64_t)a.nh, (cuuint64_t)a.R, 2};
        cuuint64_t strides[3] = {(cuuint64_t)a.d * 2, (cuuint64_t)a.nh * a.d * 2, (cuuint64_t)a.R * a.nh * a.d * 2};
        cuuint32_t box[4] = {64, 1, TC_BM, 1};
        cuuint32_t es[4] = {1, 1, 1, 1};
        if (enc(&mq, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, (void *)a.Qs, dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    const int S = a.wsplit > 1 ? a.wsplit : 1;
    o1_launch_chained(a.chain_early, k_near_tc, dim3((a.R + TC_BM - 1) / TC_BM, a.nh, S), dim3(TC_THREADS), smem, st, a, mk, mv, mq,
                      NXp, nslot);
    return cudaGetLastError();
}
