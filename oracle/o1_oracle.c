/*
 * Serial CPU oracle of a sealed O(1) attention layer: sinks, a ring-buffer
 * sliding window and a landmark far field.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path links, loads or calls
 * this file: only the tests, the smoke check and the benchmark's CPU-baseline
 * leg do. It shares no code, header, table or constant with the CUDA library.
 *
 * What it computes follows "cortiq-engine 0.8.51 src/gpu_wgpu/o1_batch.rs"
 * (module doc: a sealed layer is "rope, far insert, ring push, attend, gate,
 * blit", one row at a time, each row depending on the state the previous row
 * left), with the per-step arithmetic read off that page's kernels
 * (o1b_far_e, o1b_attend, o1b_far_commit, o1b_ring_commit, o1b_meta), the
 * rotation and table of "cortiq-engine 0.8.77 src/gpu_wgpu/dory.rs"
 * (dory_prep; the rotary table built in `run`) and the output gate of the
 * same page (dory_gate1). Everything is done one row at a time, in order,
 * in double precision, with no blocking or reordering: the state after each
 * row is exactly what the next row starts from.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  - inv[j] = base^(-2j/d) for j < d/2, rounded to f32 (the pages keep an f32
 *    inverse-frequency array but never define it); base 0 turns rotation off.
 *  - The rotary cos/sin are computed in double from the f32 frequency and
 *    stored as f32, as the pages' table is; the rotation itself is in double.
 *  - Sinks, landmark keys kt, landmark queries qt and mu are inputs, already
 *    rotated; their seal-time construction is not on the pages.
 *  - An empty far field is M = -inf, Z = 0, T = 0; the rescale factor is 1
 *    when the max does not move (including -inf == -inf).
 *  - gate == NULL means no output gate.
 *
 * Parity pins (checked by the CPU test suite, none of them by re-running this
 * file's own formulas): exact softmax attention while nothing was evicted;
 * brute force of the far algebra on tiny shapes (no running max, no ring);
 * the unit-kernel closed form; recomputation of M, Z, T from the evicted
 * keys; the meta closed form; rotation worked values and invariants; the
 * forced far-field branches.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int32_t groups;     /* G: KV groups */
    int32_t hpg;        /* query heads per group */
    int32_t d, dv;      /* key and value widths */
    int32_t sinks;      /* ns */
    int32_t window;     /* w: ring stride (the widest group window) */
    int32_t landmarks;  /* m */
    int32_t rect;       /* rectified far mass: u_b = max(u_b, 0) */
    float scale;        /* score scale (1/sqrt(d) by default) */
    float rope_base;    /* rotary base; 0 = no rotation */
} oo_geom;

/* The layer state, all arrays owned by the caller:
 *   meta   int32 [G][4]  len, head, farl, group window
 *   pos    int64 [1]     absolute position of the next row
 *   ring_k double [G][w][d], ring_v double [G][w][dv]   (rotated keys)
 *   sink_k double [G][ns][d], sink_v double [G][ns][dv]
 *   kt     double [G][m][d]          landmark keys, per group
 *   qt     double [G][hpg][m][d]     landmark queries, per head
 *   mu     double [G*hpg][m][m]      mu[a][b]: a = landmark key, b = query
 *   M, Z   double [G*hpg][m]         far max and mass
 *   T      double [G*hpg][m][dv]     far value sum                        */
typedef struct {
    int32_t *meta;
    int64_t *pos;
    double *ring_k, *ring_v;
    const double *sink_k, *sink_v, *kt, *qt, *mu;
    double *M, *Z, *T;
} oo_state;

/* Optional per-(row, head) diagnostics: the far-field sign decision and its
 * margin, so that rows whose decision sits within rounding of zero can be
 * told apart, and the denominator, whose size against sum_b |gain_b Z_b|
 * says how much a relative error in the far terms grows in the output.
 * Any pointer may be NULL. */
typedef struct {
    int8_t *have;     /* [rows][nh] 1 if the far part was kept          */
    double *far_den;  /* [rows][nh] D before the sign test (e^-c units)  */
    double *far_abs;  /* [rows][nh] sum_b |gain_b Z_b| (e^-c units)      */
    double *den;      /* [rows][nh] the row's denominator after the floor  */
} oo_diag;

/* Rotary table for one position: cs[j], sn[j], j < d/2, both rounded to f32
 * after a double evaluation of the angle p * inv[j]. */
static void oo_rope_table(int d, int64_t p, float base, double *cs, double *sn)
{
    int half = d / 2;
    for (int j = 0; j < half; j++) {
        float inv = (float)pow((double)base, -2.0 * (double)j / (double)d);
        double ang = (double)p * (double)inv;
        cs[j] = (double)(float)cos(ang);
        sn[j] = (double)(float)sin(ang);
    }
}

/* Element j pairs with j + d/2: x' = x cos - y sin, y' = y cos + x sin. */
static void oo_rotate(int d, const float *x, const double *cs, const double *sn,
                      int rotate, double *out)
{
    int half = d / 2;
    if (!rotate) {
        for (int j = 0; j < d; j++) out[j] = (double)x[j];
        return;
    }
    for (int j = 0; j < half; j++) {
        double a = (double)x[j], b = (double)x[j + half];
        out[j] = a * cs[j] - b * sn[j];
        out[j + half] = b * cs[j] + a * sn[j];
    }
}

/* Exposed for the rotation pins. */
void oo_rope(int32_t d, int64_t p, float base, const float *x, double *out)
{
    double *cs = (double *)malloc(sizeof(double) * (size_t)(d / 2 + 1));
    double *sn = (double *)malloc(sizeof(double) * (size_t)(d / 2 + 1));
    oo_rope_table(d, p, base, cs, sn);
    oo_rotate(d, x, cs, sn, base != 0.0f, out);
    free(cs);
    free(sn);
}

static double oo_dot(const double *a, const double *b, int n)
{
    double s = 0.0;
    for (int i = 0; i < n; i++) s += a[i] * b[i];
    return s;
}

/* Fresh state: empty ring and far field, position pos0. */
void oo_init(const oo_geom *g, const int32_t *group_windows, int64_t pos0, oo_state *st)
{
    int G = g->groups, nh = g->groups * g->hpg, m = g->landmarks;
    for (int gi = 0; gi < G; gi++) {
        int wg = (group_windows && group_windows[gi] > 0) ? group_windows[gi] : g->window;
        st->meta[gi * 4 + 0] = 0;
        st->meta[gi * 4 + 1] = 0;
        st->meta[gi * 4 + 2] = 0;
        st->meta[gi * 4 + 3] = wg;
    }
    *st->pos = pos0;
    memset(st->ring_k, 0, sizeof(double) * (size_t)G * g->window * g->d);
    memset(st->ring_v, 0, sizeof(double) * (size_t)G * g->window * g->dv);
    for (int i = 0; i < nh * m; i++) {
        st->M[i] = -INFINITY;
        st->Z[i] = 0.0;
    }
    memset(st->T, 0, sizeof(double) * (size_t)nh * m * g->dv);
}

typedef struct {
    const oo_geom *g;
    oo_state *st;
    int grp;
    const float *q, *k, *v, *gate;
    int32_t rows;
    double *out;
    oo_diag *diag;
    int64_t pos0;
} oo_job;

/* All rows of one KV group, serially. Groups share nothing but the row
 * position, so they may run concurrently. */
static void oo_group_rows(oo_job *jb)
{
    const oo_geom *g = jb->g;
    oo_state *st = jb->st;
    const int gi = jb->grp;
    const int G = g->groups, hpg = g->hpg, nh = G * hpg;
    const int d = g->d, dv = g->dv, ns = g->sinks, w = g->window, m = g->landmarks;
    const double scale = (double)g->scale;
    const int rotate = g->rope_base != 0.0f;

    int32_t *meta = st->meta + gi * 4;
    const int wg = meta[3];
    double *rk = st->ring_k + (size_t)gi * w * d;
    double *rv = st->ring_v + (size_t)gi * w * dv;
    const double *sk = st->sink_k + (size_t)gi * ns * d;
    const double *sv = st->sink_v + (size_t)gi * ns * dv;
    const double *kt = st->kt + (size_t)gi * m * d;

    double *cs = (double *)malloc(sizeof(double) * (size_t)(d / 2 + 1));
    double *sn = (double *)malloc(sizeof(double) * (size_t)(d / 2 + 1));
    double *kr = (double *)malloc(sizeof(double) * (size_t)d);
    double *qr = (double *)malloc(sizeof(double) * (size_t)d);
    double *s = (double *)malloc(sizeof(double) * (size_t)(ns + w));
    double *f = (double *)malloc(sizeof(double) * (size_t)(m + 1));
    double *u = (double *)malloc(sizeof(double) * (size_t)(m + 1));
    double *gain = (double *)malloc(sizeof(double) * (size_t)(m + 1));
    double *num = (double *)malloc(sizeof(double) * (size_t)dv);

    for (int r = 0; r < jb->rows; r++) {
        int64_t p = jb->pos0 + r;
        oo_rope_table(d, p, g->rope_base, cs, sn);

        /* 1. rope: the row's key (this group) */
        oo_rotate(d, jb->k + ((size_t)r * G + gi) * d, cs, sn, rotate, kr);
        const float *vrow = jb->v + ((size_t)r * G + gi) * dv;

        int len = meta[0], head = meta[1], farl = meta[2];

        /* 2. far insert: a full ring gives up its oldest key (slot head) to
         *    the far field of every head and landmark query of the group. */
        if (len == wg) {
            const double *ke = rk + (size_t)head * d;
            const double *ve = rv + (size_t)head * dv;
            for (int h = 0; h < hpg; h++) {
                int gh = gi * hpg + h;
                for (int b = 0; b < m; b++) {
                    const double *qtb = st->qt + ((size_t)gh * m + b) * d;
                    double l = scale * oo_dot(qtb, ke, d);
                    double Mo = st->M[gh * m + b];
                    double Mn = l > Mo ? l : Mo;
                    double rho = (Mn == Mo) ? 1.0 : exp(Mo - Mn);
                    double e = exp(l - Mn);
                    st->Z[gh * m + b] = st->Z[gh * m + b] * rho + e;
                    double *Tb = st->T + ((size_t)gh * m + b) * dv;
                    for (int t = 0; t < dv; t++) Tb[t] = Tb[t] * rho + e * ve[t];
                    st->M[gh * m + b] = Mn;
                }
            }
            farl += 1;
        }

        /* 3. ring push: slot (head + len) % wg, which is the evicted slot when
         *    the ring was full. */
        {
            int slot = (head + len) % wg;
            memcpy(rk + (size_t)slot * d, kr, sizeof(double) * (size_t)d);
            for (int t = 0; t < dv; t++) rv[(size_t)slot * dv + t] = (double)vrow[t];
            if (len == wg) head = (head + 1) % wg;
            else len += 1;
        }
        meta[0] = len;
        meta[1] = head;
        meta[2] = farl;

        /* 4. attend, per query head of the group */
        for (int h = 0; h < hpg; h++) {
            int gh = gi * hpg + h;
            oo_rotate(d, jb->q + ((size_t)r * nh + gh) * d, cs, sn, rotate, qr);

            int n = ns + len;
            double c0 = -INFINITY;
            for (int x = 0; x < ns; x++) {
                s[x] = scale * oo_dot(qr, sk + (size_t)x * d, d);
                if (s[x] > c0) c0 = s[x];
            }
            for (int x = 0; x < len; x++) {
                int slot = (head + x) % wg;
                s[ns + x] = scale * oo_dot(qr, rk + (size_t)slot * d, d);
                if (s[ns + x] > c0) c0 = s[ns + x];
            }

            double c = c0, D = 0.0, Dabs = 0.0;
            int have = 0;
            if (farl > 0) {
                double F = -INFINITY;
                for (int a = 0; a < m; a++) {
                    f[a] = scale * oo_dot(qr, kt + (size_t)a * d, d);
                    if (f[a] > F) F = f[a];
                }
                const double *mu = st->mu + (size_t)gh * m * m;
                for (int b = 0; b < m; b++) {
                    double acc = 0.0;
                    for (int a = 0; a < m; a++) acc += exp(f[a] - F) * mu[(size_t)a * m + b];
                    if (g->rect && acc < 0.0) acc = 0.0;
                    u[b] = acc;
                }
                for (int b = 0; b < m; b++) {
                    double cb = F + st->M[gh * m + b];
                    if (cb > c) c = cb;
                }
                for (int b = 0; b < m; b++) {
                    gain[b] = u[b] * exp(F + st->M[gh * m + b] - c);
                    D += gain[b] * st->Z[gh * m + b];
                    Dabs += fabs(gain[b] * st->Z[gh * m + b]);
                }
                if (D >= 0.0) have = 1;
            }
            if (jb->diag) {
                size_t at = (size_t)r * nh + gh;
                if (jb->diag->have) jb->diag->have[at] = (int8_t)have;
                if (jb->diag->far_den) jb->diag->far_den[at] = D;
                if (jb->diag->far_abs) jb->diag->far_abs[at] = Dabs;
            }
            if (!have) D = 0.0;

            double den = D;
            for (int t = 0; t < dv; t++) num[t] = 0.0;
            if (have) {
                for (int b = 0; b < m; b++) {
                    const double *Tb = st->T + ((size_t)gh * m + b) * dv;
                    for (int t = 0; t < dv; t++) num[t] += gain[b] * Tb[t];
                }
            }
            for (int x = 0; x < n; x++) {
                double pw = exp(s[x] - c);
                den += pw;
                const double *vx = (x < ns) ? sv + (size_t)x * dv
                                            : rv + (size_t)((head + (x - ns)) % wg) * dv;
                for (int t = 0; t < dv; t++) num[t] += pw * vx[t];
            }
            if (den < 1e-30) den = 1e-30;
            if (jb->diag && jb->diag->den) jb->diag->den[(size_t)r * nh + gh] = den;

            /* 5. gate, and the row's output */
            double *o = jb->out + ((size_t)r * nh + gh) * dv;
            for (int t = 0; t < dv; t++) {
                double y = num[t] / den;
                if (jb->gate) {
                    double gl = (double)jb->gate[((size_t)r * nh + gh) * dv + t];
                    y = y / (1.0 + exp(-gl));
                }
                o[t] = y;
            }
        }
    }
    free(cs); free(sn); free(kr); free(qr); free(s); free(f); free(u); free(gain); free(num);
}

static void *oo_thread(void *arg)
{
    oo_group_rows((oo_job *)arg);
    return NULL;
}

/* `rows` consecutive rows through the layer. q [rows][G*hpg][d], k [rows][G][d],
 * v [rows][G][dv], gate [rows][G*hpg][dv] or NULL; out [rows][G*hpg][dv].
 * KV groups run on up to `threads` threads; the rows of a group are serial.
 * Returns the number of threads used. */
int32_t oo_rows(const oo_geom *g, oo_state *st, const float *q, const float *k,
                const float *v, const float *gate, int32_t rows, double *out,
                oo_diag *diag, int32_t threads)
{
    int G = g->groups;
    oo_job *jobs = (oo_job *)calloc((size_t)G, sizeof(oo_job));
    for (int gi = 0; gi < G; gi++) {
        jobs[gi].g = g;
        jobs[gi].st = st;
        jobs[gi].grp = gi;
        jobs[gi].q = q;
        jobs[gi].k = k;
        jobs[gi].v = v;
        jobs[gi].gate = gate;
        jobs[gi].rows = rows;
        jobs[gi].out = out;
        jobs[gi].diag = diag;
        jobs[gi].pos0 = *st->pos;
    }
    int used = 1;
    if (threads > 1 && G > 1) {
        int nt = threads < G ? threads : G;
        pthread_t *tid = (pthread_t *)calloc((size_t)G, sizeof(pthread_t));
        for (int base = 0; base < G; base += nt) {
            int hi = base + nt < G ? base + nt : G;
            for (int gi = base; gi < hi; gi++) pthread_create(&tid[gi], NULL, oo_thread, &jobs[gi]);
            for (int gi = base; gi < hi; gi++) pthread_join(tid[gi], NULL);
        }
        free(tid);
        used = nt;
    } else {
        for (int gi = 0; gi < G; gi++) oo_group_rows(&jobs[gi]);
    }
    *st->pos += rows;
    free(jobs);
    return used;
}

/* Rewind `rows` pushes of every group's ring ("cortiq-engine 0.8.77
 * src/gpu_wgpu/dory.rs", dory_o1_back, the looped-layer KV mode's rewind),
 * one row at a time as the page does it: a full ring (len == wg) steps its
 * head back by one and forgets one eviction (farl - 1); a ring not yet full
 * drops its newest entry (len - 1). Ring contents and the far field (M, Z,
 * T) are not undone, as on the page. The position moves back by `rows`.
 * Reading where the page is silent: a rewind no group can take in full
 * (len < rows while not full, farl < rows while full, or pos < rows) is
 * refused before anything changes. Returns 0, or -1 when refused. */
int32_t oo_back(const oo_geom *g, oo_state *st, int32_t rows)
{
    if (rows < 0 || *st->pos < rows) return -1;
    for (int gi = 0; gi < g->groups; gi++) {
        const int32_t *mt = st->meta + 4 * gi;
        if (mt[0] == mt[3] ? mt[2] < rows : mt[0] < rows) return -1;
    }
    for (int gi = 0; gi < g->groups; gi++) {
        int32_t *mt = st->meta + 4 * gi;
        for (int r = 0; r < rows; r++) {
            const int32_t wg = mt[3];
            if (mt[0] == wg) {
                mt[1] = (mt[1] + wg - 1) % wg;
                mt[2] -= 1;
            } else {
                mt[0] -= 1;
            }
        }
    }
    *st->pos -= rows;
    return 0;
}

