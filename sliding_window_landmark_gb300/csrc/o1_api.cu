// The C ABI of include/o1.h: argument validation, the state header, the
// pass loop of o1_chunk_attend, and host snapshots. Every check runs before
// any launch; nothing here falls back to another implementation.
#include <math.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <unordered_map>

#include "o1_common.cuh"

// Scratch of o1_token_attend_noalloc: a file-scope device array, so that the
// entry point allocates nothing. Every call on a device shares it.
static __device__ __align__(256) unsigned char o1_noalloc_scratch[O1_NOALLOC_SCRATCH_BYTES];

extern const char *const o1_stage_names[O1_NUM_STAGES];

namespace {

// Limit of the kernels' first waits for calls launched from now on
// (o1_set_wait_limit); drains of work already in flight keep the full limit.
std::atomic<long long> g_wait_cycles{O1_WAIT_CYCLES_FULL};

bool geom_ok(const o1_geom *g) {
    if (!g) return false;
    if (g->groups < 1 || g->groups > 4096) return false;
    if (g->heads_per_group < 1 || g->heads_per_group > O1_MAX_HPG) return false;
    if (g->d < 8 || g->d > O1_MAX_D || g->d % 8) return false;
    if (g->dv < 4 || g->dv > O1_MAX_DV || g->dv % 4) return false;
    if (g->sinks < 0 || g->sinks > O1_MAX_NS) return false;
    if (g->window < 1 || g->window > O1_MAX_W) return false;
    if (g->landmarks < 1 || g->landmarks > O1_MAX_M) return false;
    if (!(g->scale == g->scale) || !isfinite(g->scale)) return false;
    if (!isfinite(g->rope_base) || g->rope_base < 0.f) return false;
    if (g->rect_far_mass != 0 && g->rect_far_mass != 1) return false;
    return true;
}

bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

// Largest pass (rows) whose scratch fits in `bytes`.
int scratch_cap(const o1_geom &g, size_t bytes) {
    if (o1_scratch_layout(g, 1).total > bytes) return 0;
    int lo = 1, hi = 1 << 24;
    while (lo < hi) {
        const int mid = lo + (hi - lo + 1) / 2;
        if (o1_scratch_layout(g, mid).total <= bytes) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

O1Args state_args(void *state, const o1_geom &g) {
    const O1Layout L = o1_layout(g);
    char *b = (char *)state;
    O1Args a;
    memset(&a, 0, sizeof(a));
    a.commit = 1;
    a.wait_cycles = g_wait_cycles.load(std::memory_order_relaxed);
    a.G = g.groups;
    a.hpg = g.heads_per_group;
    a.nh = g.groups * g.heads_per_group;
    a.d = g.d;
    a.dv = g.dv;
    a.ns = g.sinks;
    a.w = g.window;
    a.m = g.landmarks;
    a.rect = g.rect_far_mass;
    a.rotate = g.rope_base != 0.f;
    a.scale = g.scale;
    a.hdr = (O1Header *)(b + L.hdr);
    a.meta = (uint32_t *)(b + L.meta);
    a.ring_k = (float *)(b + L.ring_k);
    a.ring_v = (float *)(b + L.ring_v);
    a.sink_k = (const float *)(b + L.sink_k);
    a.sink_v = (const float *)(b + L.sink_v);
    a.kt = (const float *)(b + L.kt);
    a.qt = (const float *)(b + L.qt);
    a.mu = (const float *)(b + L.mu);
    a.M = (float *)(b + L.M);
    a.Z = (float *)(b + L.Z);
    a.Zlo = (float *)(b + L.Zlo);
    a.T = (float *)(b + L.T);
    a.tick = (uint32_t *)(b + L.tick);
    return a;
}

void scratch_args(O1Args &a, void *scratch, const O1Scratch &S) {
    char *b = (char *)scratch;
    a.qr = (float *)(b + S.qr);
    a.kr = (float *)(b + S.kr);
    a.E = (float *)(b + S.E);
    a.P = (float *)(b + S.P);
    a.Fb = (float *)(b + S.Fb);
    a.Tp = (float *)(b + S.Tp);
    a.fh = (float *)(b + S.fh);
    a.sh = (float *)(b + S.sh);
    a.sn = (float *)(b + S.sn);
    a.cap = S.ldc;   // the row stride of E and P
    a.Xk = (unsigned short *)(b + S.Xk);
    a.XvT = (unsigned short *)(b + S.XvT);
    a.Qs = (unsigned short *)(b + S.Qs);
    a.nxp = S.nxp;
    a.tc = S.nxp > 0;
    a.Sp = S.cap >= 2 ? (float *)(b + S.Sp) : nullptr;
    a.wpart = (float *)(b + S.Wp);
}

// The state the last one-row step on each stream was launched on. A step on
// the same state right after it would find the copies it issues before its
// wait stale (the kernel checks and fetches again), so it issues them after
// the wait instead. Only a choice of timing: the kernel's own check of the
// position is what keeps the copies correct.
int tok_prefetch_for(cudaStream_t st, const void *state) {
    static std::mutex mu;
    static std::unordered_map<const void *, const void *> last;
    std::lock_guard<std::mutex> lock(mu);
    const void *&prev = last[(const void *)st];
    const int prefetch = prev != state;
    prev = state;
    return prefetch;
}

int chunk(void *state, const o1_geom *geom, void *scratch, size_t scratch_bytes, const float *q,
          const float *k, const float *v, const float *gate, int32_t rows, float *out, void *stream,
          cudaEvent_t const *ev = nullptr, int commit = 1, int exact = 0) {
    if (!geom_ok(geom)) return O1_ERR_UNSUPPORTED;
    if (rows < 0) return O1_ERR_ARG;
    if (rows == 0) return O1_OK;
    if (!state || !scratch || !q || !k || !v || !out) return O1_ERR_ARG;
    if (!aligned(state, 256) || !aligned(scratch, 256)) return O1_ERR_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
        (gate && !aligned(gate, 16)))
        return O1_ERR_ARG;
    const o1_geom &g = *geom;
    const size_t nh = (size_t)g.groups * g.heads_per_group;
    // out must not overlap an input: the near kernel reads gate while writing out
    const char *ob = (const char *)out, *oe = ob + (size_t)rows * nh * g.dv * 4;
    auto overlaps = [&](const void *p, size_t n) {
        const char *pb = (const char *)p, *pe = pb + n;
        return p && pb < oe && ob < pe;
    };
    if (overlaps(q, (size_t)rows * nh * g.d * 4) || overlaps(k, (size_t)rows * g.groups * g.d * 4) ||
        overlaps(v, (size_t)rows * g.groups * g.dv * 4) || overlaps(gate, (size_t)rows * nh * g.dv * 4))
        return O1_ERR_ARG;
    const int cap = scratch_cap(g, scratch_bytes);
    if (cap < 1 || scratch_bytes < o1_tok_layout(g).total) return O1_ERR_ARG;
    // attend-only calls run as one pass: a later pass would need the state
    // the earlier one leaves
    if (!commit && rows > cap) return O1_ERR_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    O1Args a = state_args(state, g);
    a.commit = commit;
    a.exact = exact;
    for (int r0 = 0; r0 < rows; r0 += cap) {
        const int R = rows - r0 < cap ? rows - r0 : cap;
        if (R == 1 && !ev && commit) {
            // one row: the decode path
            const O1TokScratch T = o1_tok_layout(g);
            char *sb = (char *)scratch;
            a.part = (float *)(sb + T.part);
            a.pml = (float *)(sb + T.pml);
            a.farp = (float *)(sb + T.farp);
            a.kcur = (float *)(sb + T.kcur);
            a.KC = T.KC;
            a.NC = T.NC;
            a.NF = T.NF;
            a.MB = T.MB;
            a.tok_smem = T.smem;
            a.tok_prefetch = tok_prefetch_for(st, state);
            a.q = q + (size_t)r0 * nh * g.d;
            a.k = k + (size_t)r0 * g.groups * g.d;
            a.v = v + (size_t)r0 * g.groups * g.dv;
            a.gate = gate ? gate + (size_t)r0 * nh * g.dv : nullptr;
            a.out = out + (size_t)r0 * nh * g.dv;
            a.R = 1;
            const cudaError_t te = o1_launch_token(a, st);
            if (te == cudaSuccess) continue;
            // cudaErrorInvalidConfiguration: the one-row kernel's shared
            // memory exceeds a block's for this geometry (windows of a few
            // hundred thousand keys); the row takes a one-row pass instead
            if (te != cudaErrorInvalidConfiguration) return O1_ERR_CUDA;
        }
        const O1Scratch S = o1_scratch_layout(g, R);
        scratch_args(a, scratch, S);
        a.q = q + (size_t)r0 * nh * g.d;
        a.k = k + (size_t)r0 * g.groups * g.d;
        a.v = v + (size_t)r0 * g.groups * g.dv;
        a.gate = gate ? gate + (size_t)r0 * nh * g.dv : nullptr;
        a.out = out + (size_t)r0 * nh * g.dv;
        a.R = R;
        a.nsub = S.nsub;
        if (o1_launch_pass(a, st, ev) != cudaSuccess) return O1_ERR_CUDA;
    }
    return O1_OK;
}

int check_header(const void *state, const o1_geom &g, cudaStream_t st) {
    O1Header h;
    if (cudaMemcpyAsync(&h, state, sizeof(h), cudaMemcpyDeviceToHost, st) != cudaSuccess) return O1_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return O1_ERR_CUDA;
    if (h.magic != O1_MAGIC || h.version != O1_VERSION || memcmp(&h.geom, &g, sizeof(o1_geom)) != 0)
        return O1_ERR_STATE;
    return O1_OK;
}

// Device address of o1_noalloc_scratch on the current device, looked up once
// per device. In host code the array's name is only a host-side stand-in,
// never a device address.
int noalloc_scratch(void **out) {
    static std::mutex mu;
    static void *addr[256];
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return O1_ERR_CUDA;
    if (dev < 0 || dev >= 256) return O1_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, o1_noalloc_scratch) != cudaSuccess || !p) return O1_ERR_CUDA;
        addr[dev] = p;
    }
    *out = addr[dev];
    return O1_OK;
}

}  // namespace

extern "C" {

size_t o1_state_bytes(const o1_geom *geom) {
    if (!geom_ok(geom)) return 0;
    return o1_layout(*geom).total;
}

size_t o1_scratch_bytes(const o1_geom *geom, int32_t max_rows) {
    if (!geom_ok(geom) || max_rows < 1) return 0;
    return o1_scratch_need(*geom, max_rows);
}

int o1_state_init(void *state, const o1_geom *geom, const int32_t *group_windows, const float *sink_k,
                  const float *sink_v, const float *k_tilde, const float *q_tilde, const float *mu, int64_t pos0,
                  void *stream) {
    if (!geom_ok(geom)) return O1_ERR_UNSUPPORTED;
    const o1_geom &g = *geom;
    if (!state || !aligned(state, 256) || !k_tilde || !q_tilde || !mu) return O1_ERR_ARG;
    if (g.sinks > 0 && (!sink_k || !sink_v)) return O1_ERR_ARG;
    if (pos0 < 0) return O1_ERR_ARG;
    if (group_windows)
        for (int i = 0; i < g.groups; ++i)
            if (group_windows[i] < 0 || group_windows[i] > g.window) return O1_ERR_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    const O1Layout L = o1_layout(g);
    const size_t G = g.groups, nh = G * g.heads_per_group, m = g.landmarks;

    O1Header h;
    memset(&h, 0, sizeof(h));
    h.magic = O1_MAGIC;
    h.version = O1_VERSION;
    h.geom = g;
    h.pos = pos0;
    h.ticket = 0;
    // inv[j] = base^(-2j/d), rounded to f32
    for (int j = 0; j < g.d / 2; ++j)
        h.inv_freq[j] = g.rope_base != 0.f ? (float)pow((double)g.rope_base, -2.0 * j / (double)g.d) : 0.f;
    uint32_t meta[4 * 4096];
    for (int i = 0; i < g.groups; ++i) {
        const int wg = (group_windows && group_windows[i] > 0) ? group_windows[i] : g.window;
        meta[i * 4 + 0] = 0;
        meta[i * 4 + 1] = 0;
        meta[i * 4 + 2] = 0;
        meta[i * 4 + 3] = (uint32_t)wg;
    }
    char *b = (char *)state;
    cudaError_t e = cudaSuccess;
    auto cp = [&](size_t off, const void *src, size_t n, cudaMemcpyKind kind) {
        if (e == cudaSuccess && n) e = cudaMemcpyAsync(b + off, src, n, kind, st);
    };
    cp(L.hdr, &h, sizeof(h), cudaMemcpyHostToDevice);
    cp(L.meta, meta, G * 4 * sizeof(uint32_t), cudaMemcpyHostToDevice);
    cp(L.sink_k, sink_k, G * g.sinks * g.d * 4, cudaMemcpyDeviceToDevice);
    cp(L.sink_v, sink_v, G * g.sinks * g.dv * 4, cudaMemcpyDeviceToDevice);
    cp(L.kt, k_tilde, G * m * g.d * 4, cudaMemcpyDeviceToDevice);
    cp(L.qt, q_tilde, nh * m * g.d * 4, cudaMemcpyDeviceToDevice);
    cp(L.mu, mu, nh * m * m * 4, cudaMemcpyDeviceToDevice);
    if (e != cudaSuccess) return O1_ERR_CUDA;
    // the header and meta come from this stack frame: finish those copies
    if (cudaStreamSynchronize(st) != cudaSuccess) return O1_ERR_CUDA;
    O1Args a = state_args(state, g);
    if (o1_launch_init(a, st) != cudaSuccess) return O1_ERR_CUDA;
    return O1_OK;
}

int o1_chunk_attend(void *state, const o1_geom *geom, void *scratch, size_t scratch_bytes, const float *q,
                    const float *k, const float *v, const float *gate, int32_t rows, float *out, void *stream) {
    return chunk(state, geom, scratch, scratch_bytes, q, k, v, gate, rows, out, stream);
}

int o1_chunk_attend_timed(void *state, const o1_geom *geom, void *scratch, size_t scratch_bytes,
                          const float *q, const float *k, const float *v, const float *gate, int32_t rows,
                          float *out, void *const *events, int32_t n_events, void *stream) {
    if (!events || n_events < 2 * O1_NUM_STAGES) return O1_ERR_ARG;
    for (int i = 0; i < 2 * O1_NUM_STAGES; ++i)
        if (!events[i]) return O1_ERR_ARG;
    return chunk(state, geom, scratch, scratch_bytes, q, k, v, gate, rows, out, stream,
                 (cudaEvent_t const *)events);
}

int o1_chunk_attend_spec(void *state, const o1_geom *geom, void *scratch, size_t scratch_bytes, const float *q,
                         const float *k, const float *v, const float *gate, int32_t rows, float *out,
                         void *stream) {
    return chunk(state, geom, scratch, scratch_bytes, q, k, v, gate, rows, out, stream, nullptr, 0);
}

int o1_window_attend(void *state, const o1_geom *geom, void *scratch, size_t scratch_bytes, const float *q,
                     const float *k, const float *v, const float *gate, int32_t rows, float *out, void *stream) {
    return chunk(state, geom, scratch, scratch_bytes, q, k, v, gate, rows, out, stream, nullptr, 0, 1);
}

int o1_spec_commit(void *state, const o1_geom *geom, void *scratch, size_t scratch_bytes, const float *k,
                   const float *v, int32_t rows, void *stream) {
    if (!geom_ok(geom)) return O1_ERR_UNSUPPORTED;
    if (rows < 0) return O1_ERR_ARG;
    if (rows == 0) return O1_OK;
    if (!state || !scratch || !k || !v) return O1_ERR_ARG;
    if (!aligned(state, 256) || !aligned(scratch, 256) || !aligned(k, 16) || !aligned(v, 16)) return O1_ERR_ARG;
    const o1_geom &g = *geom;
    const int cap = scratch_cap(g, scratch_bytes);
    if (cap < 1 || scratch_bytes < o1_tok_layout(g).total) return O1_ERR_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    O1Args a = state_args(state, g);
    if (rows == 1) {
        // one row: the one-row kernel's far chunks insert the evicted key and
        // the last of them commits; nothing attends
        const O1TokScratch T = o1_tok_layout(g);
        char *sb = (char *)scratch;
        a.part = (float *)(sb + T.part);
        a.pml = (float *)(sb + T.pml);
        a.farp = (float *)(sb + T.farp);
        a.kcur = (float *)(sb + T.kcur);
        a.KC = T.KC;
        a.NC = T.NC;
        a.NF = T.NF;
        a.MB = T.MB;
        a.tok_smem = T.smem;
        a.tok_prefetch = tok_prefetch_for(st, state);
        a.tok_commit_only = 1;
        a.k = k;
        a.v = v;
        a.R = 1;
        const cudaError_t te = o1_launch_token(a, st);
        if (te == cudaSuccess) return O1_OK;
        // the one-row kernel does not fit this geometry: a one-row commit pass
        if (te != cudaErrorInvalidConfiguration) return O1_ERR_CUDA;
        a = state_args(state, g);
    }
    for (int r0 = 0; r0 < rows; r0 += cap) {
        const int R = rows - r0 < cap ? rows - r0 : cap;
        const O1Scratch S = o1_scratch_layout(g, R);
        scratch_args(a, scratch, S);
        a.tc = 0;   // no window attention in this pass
        a.q = nullptr;
        a.k = k + (size_t)r0 * g.groups * g.d;
        a.v = v + (size_t)r0 * g.groups * g.dv;
        a.gate = nullptr;
        a.out = nullptr;
        a.R = R;
        a.nsub = S.nsub;
        if (o1_launch_commit_pass(a, st) != cudaSuccess) return O1_ERR_CUDA;
    }
    return O1_OK;
}

int o1_state_back(void *state, const o1_geom *geom, int32_t rows, void *stream) {
    if (!geom_ok(geom)) return O1_ERR_UNSUPPORTED;
    if (!state || !aligned(state, 256) || rows < 0) return O1_ERR_ARG;
    if (rows == 0) return O1_OK;
    const O1Args a = state_args(state, *geom);
    return o1_launch_back(a, rows, (cudaStream_t)stream) == cudaSuccess ? O1_OK : O1_ERR_CUDA;
}

const char *o1_stage_name(int32_t stage) {
    return (stage >= 0 && stage < O1_NUM_STAGES) ? o1_stage_names[stage] : nullptr;
}

int o1_token_attend(void *state, const o1_geom *geom, void *scratch, size_t scratch_bytes, const float *q,
                    const float *k, const float *v, const float *gate, float *out, void *stream) {
    return chunk(state, geom, scratch, scratch_bytes, q, k, v, gate, 1, out, stream);
}

int o1_token_attend_noalloc(void *state, const o1_geom *geom, const float *q, const float *k, const float *v,
                            const float *gate, float *out, void *stream) {
    if (!geom_ok(geom)) return O1_ERR_UNSUPPORTED;
    if (o1_scratch_need(*geom, 1) > (size_t)O1_NOALLOC_SCRATCH_BYTES) return O1_ERR_UNSUPPORTED;
    if (!state || !q || !k || !v || !out) return O1_ERR_ARG;
    void *scratch = nullptr;
    const int st = noalloc_scratch(&scratch);
    if (st != O1_OK) return st;
    return chunk(state, geom, scratch, O1_NOALLOC_SCRATCH_BYTES, q, k, v, gate, 1, out, stream);
}

int o1_state_read(const void *state, const o1_geom *geom, o1_state_host *dst, void *stream) {
    if (!geom_ok(geom)) return O1_ERR_UNSUPPORTED;
    if (!state || !dst || !aligned(state, 256)) return O1_ERR_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    const int hs = check_header(state, *geom, st);
    if (hs != O1_OK) return hs;
    const o1_geom &g = *geom;
    const O1Layout L = o1_layout(g);
    const size_t G = g.groups, nh = G * g.heads_per_group, m = g.landmarks;
    const char *b = (const char *)state;
    cudaError_t e = cudaSuccess;
    auto cp = [&](void *dstp, size_t off, size_t n) {
        if (e == cudaSuccess && dstp && n) e = cudaMemcpyAsync(dstp, b + off, n, cudaMemcpyDeviceToHost, st);
    };
    cp(dst->meta, L.meta, G * 4 * sizeof(uint32_t));
    cp(dst->pos, L.hdr + offsetof(O1Header, pos), sizeof(int64_t));
    cp(dst->ring_k, L.ring_k, G * g.window * g.d * 4);
    cp(dst->ring_v, L.ring_v, G * g.window * g.dv * 4);
    cp(dst->far_max, L.M, nh * m * 4);
    cp(dst->far_mass, L.Z, nh * m * 4);
    cp(dst->far_val, L.T, nh * m * g.dv * 4);
    if (e != cudaSuccess) return O1_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return O1_ERR_CUDA;
    return O1_OK;
}

int o1_state_write(void *state, const o1_geom *geom, const o1_state_host *src, void *stream) {
    if (!geom_ok(geom)) return O1_ERR_UNSUPPORTED;
    if (!state || !src || !aligned(state, 256)) return O1_ERR_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    const int hs = check_header(state, *geom, st);
    if (hs != O1_OK) return hs;
    const o1_geom &g = *geom;
    if (src->meta)
        for (int i = 0; i < g.groups; ++i) {
            const uint32_t len = src->meta[i * 4], head = src->meta[i * 4 + 1], wg = src->meta[i * 4 + 3];
            if (wg < 1 || wg > (uint32_t)g.window || len > wg || head >= wg) return O1_ERR_ARG;
        }
    if (src->pos && *src->pos < 0) return O1_ERR_ARG;
    const O1Layout L = o1_layout(g);
    const size_t G = g.groups, nh = G * g.heads_per_group, m = g.landmarks;
    char *b = (char *)state;
    cudaError_t e = cudaSuccess;
    auto cp = [&](const void *srcp, size_t off, size_t n) {
        if (e == cudaSuccess && srcp && n) e = cudaMemcpyAsync(b + off, srcp, n, cudaMemcpyHostToDevice, st);
    };
    cp(src->meta, L.meta, G * 4 * sizeof(uint32_t));
    cp(src->pos, L.hdr + offsetof(O1Header, pos), sizeof(int64_t));
    cp(src->ring_k, L.ring_k, G * g.window * g.d * 4);
    cp(src->ring_v, L.ring_v, G * g.window * g.dv * 4);
    cp(src->far_max, L.M, nh * m * 4);
    cp(src->far_mass, L.Z, nh * m * 4);
    cp(src->far_val, L.T, nh * m * g.dv * 4);
    // a written far mass is exact as given: its low part is zero
    if (e == cudaSuccess && src->far_mass) e = cudaMemsetAsync(b + L.Zlo, 0, nh * m * 4, st);
    if (e != cudaSuccess) return O1_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return O1_ERR_CUDA;
    return O1_OK;
}

int o1_state_flags(void *state, const o1_geom *geom, uint32_t *flags, int32_t clear, void *stream) {
    if (!geom_ok(geom)) return O1_ERR_UNSUPPORTED;
    if (!state || !flags || !aligned(state, 256)) return O1_ERR_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    const int hs = check_header(state, *geom, st);
    if (hs != O1_OK) return hs;
    char *b = (char *)state + o1_layout(*geom).hdr + offsetof(O1Header, flags);
    if (cudaMemcpyAsync(flags, b, sizeof(uint32_t), cudaMemcpyDeviceToHost, st) != cudaSuccess) return O1_ERR_CUDA;
    if (clear && cudaMemsetAsync(b, 0, sizeof(uint32_t), st) != cudaSuccess) return O1_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return O1_ERR_CUDA;
    return O1_OK;
}

int o1_set_wait_limit(int64_t cycles) {
    g_wait_cycles.store(cycles < 1 || cycles > O1_WAIT_CYCLES_FULL ? O1_WAIT_CYCLES_FULL : (long long)cycles,
                        std::memory_order_relaxed);
    return O1_OK;
}

const char *o1_status_string(int status) {
    switch (status) {
        case O1_OK: return "ok";
        case O1_ERR_ARG: return "invalid argument (null, misaligned, overlapping or too small buffer, bad size)";
        case O1_ERR_UNSUPPORTED: return "geometry outside the library's limits";
        case O1_ERR_CUDA: return "a CUDA launch or copy failed";
        case O1_ERR_STATE: return "state header does not match the geometry";
        default: return "unknown status";
    }
}

}  // extern "C"
