/*
 * o1.h — C ABI of the sealed O(1) layer attention library (libo1.so, CUDA,
 * sm_103a).
 *
 * A sealed layer's attention: every query row attends to
 *   (1) a few sink keys,
 *   (2) a ring-buffer window of recent keys (the causal rows of the call
 *       included), and
 *   (3) a constant-size far field that summarises every key evicted from the
 *       ring: per (group, head, landmark query b) a running max M_b, mass Z_b
 *       and value sum T_b of exp(scale * qt_b . k_evicted - M_b), read back
 *       through the landmark keys kt and the coefficients mu.
 * The method is the one of "cortiq-engine 0.8.51 src/gpu_wgpu/o1_batch.rs"
 * (module doc; kernels o1b_far_e, o1b_attend, o1b_far_commit,
 * o1b_ring_commit, o1b_meta); the one-row variant is the one of
 * "cortiq-engine 0.8.82 src/gpu_metal/o1c.rs" (encode_tok) and of
 * "cortiq-engine 0.8.77 src/gpu_wgpu/dory.rs" (dory_os ... dory_ogate), whose
 * rotation (dory_prep) and output gate (dory_gate1) it also applies.
 *
 * Conventions, for every entry point:
 *  - Ownership: the caller allocates and frees every buffer. The library
 *    allocates no device or host memory for a call; a state buffer carries
 *    its own header. What it keeps itself: the second CUDA stream and two
 *    events of the chunk path (one set per host thread and device, made by
 *    the first chunk call and released when that thread exits; see
 *    O1_NUM_STAGES) and the static scratch array of o1_token_attend_noalloc.
 *  - Pointers: "device" pointers are CUDA global memory of the current
 *    device, "host" pointers are ordinary process memory. Device buffers must
 *    be 16-byte aligned (a torch or cudaMalloc allocation always is); the
 *    state and scratch buffers 256-byte aligned.
 *  - Layouts are row-major fp32 unless stated; shapes are written [a][b][c]
 *    with the last index fastest.
 *  - Streams: `stream` is a cudaStream_t passed as void* (NULL = the legacy
 *    default stream). Calls are asynchronous on it except where stated. A
 *    state must be used from one stream at a time.
 *  - Errors: every call validates its arguments before launching anything
 *    and returns O1_OK or a negative status; nothing falls back to another
 *    implementation. O1_ERR_CUDA reports a failed launch or copy
 *    (cudaGetLastError after the launches, which also clears a launch
 *    error so that it is reported once; or the copy's status).
 *  - State and geometry: the state's header (magic, geometry) lives on the
 *    device. The calls that synchronise anyway (o1_state_read, _write,
 *    _flags) check it against `geom` and return O1_ERR_STATE on a mismatch.
 *    The attend, commit and rewind calls do not read it back: that would
 *    cost a device round trip per call and make them uncapturable. They
 *    must be given the geometry the state was initialised with.
 */
#ifndef O1_H
#define O1_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define O1_API __attribute__((visibility("default")))
#else
#define O1_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
enum {
    O1_OK = 0,
    O1_ERR_ARG = -1,          /* null or misaligned pointer, bad size        */
    O1_ERR_UNSUPPORTED = -2,  /* geometry outside the library's limits       */
    O1_ERR_CUDA = -3,         /* a CUDA launch or copy failed                */
    O1_ERR_STATE = -4         /* state header does not match the geometry    */
};

/* Geometry of one sealed layer ("cortiq-engine 0.8.51 src/gpu_wgpu/o1_batch.rs",
 * struct Geom). Limits: groups >= 1, heads_per_group in [1, 16],
 * d in [8, 256] with d % 8 == 0, dv in [4, 256] with dv % 4 == 0,
 * sinks in [0, 64], window in [1, 1 << 20], landmarks in [1, 64]. */
typedef struct o1_geom {
    int32_t groups;           /* G: KV groups                                  */
    int32_t heads_per_group;  /* hpg: query heads per KV group (nh = G * hpg)  */
    int32_t d;                /* key / query width                             */
    int32_t dv;               /* value width                                   */
    int32_t sinks;            /* ns: sink keys per group                       */
    int32_t window;           /* w: ring stride = the widest group window      */
    int32_t landmarks;        /* m: landmark queries per head                  */
    int32_t rect_far_mass;    /* 1: u_b = max(u_b, 0) (the pages' rect_fm)     */
    float scale;              /* score scale, normally 1/sqrt(d)               */
    float rope_base;          /* rotary base (e.g. 1e6); 0 = no rotation       */
} o1_geom;

/* Host-side view of a state, for o1_state_read / o1_state_write. Every
 * pointer is host memory and may be NULL (that part is skipped). */
typedef struct o1_state_host {
    uint32_t *meta;    /* [G][4]: len, head, farl, group window                */
    int64_t *pos;      /* [1]: absolute position of the next row               */
    float *ring_k;     /* [G][window][d]: rotated keys by ring slot            */
    float *ring_v;     /* [G][window][dv]                                      */
    float *far_max;    /* M [G*hpg][m]; -inf while the far field is empty      */
    float *far_mass;   /* Z [G*hpg][m], rounded to f32 (the state keeps a low
                          part beside it; a write sets that part to zero)    */
    float *far_val;    /* T [G*hpg][m][dv]                                     */
} o1_state_host;

/* Bytes of device memory a state of this geometry needs (0 if the geometry is
 * outside the limits). Host-only; no CUDA call.
 * The state holds the buffers of one sealed layer that "cortiq-engine 0.8.51
 * src/gpu_wgpu/o1_batch.rs" lists in struct State (meta, ring_k, ring_v,
 * sink_k, sink_v, k_tilde, qt, mu, the far max and mass mz, the far value
 * sum that), sized from struct Geom, plus a header of this library's
 * (magic, geometry, position, rotary frequencies, flags). */
O1_API size_t o1_state_bytes(const o1_geom *geom);

/* Bytes of device scratch that lets one o1_chunk_attend launch process up to
 * `max_rows` rows in one pass (longer calls run in passes of that many rows).
 * 0 if the geometry is unsupported or max_rows < 1. Host-only.
 * The pages size a per-call scratch from the geometry ("cortiq-engine 0.8.51
 * src/gpu_wgpu/o1_batch.rs", Geom::scratch_len: the far-field exponents and
 * prefixes of one 64-row sub-chunk plus a max and a rescale per head and
 * landmark). This library runs every 64-row block of a pass at once, so its
 * scratch holds those planes for all of them, plus the rotated rows, the
 * window and side partials and, on the tensor-core path, fp16 panels. */
O1_API size_t o1_scratch_bytes(const o1_geom *geom, int32_t max_rows);

/* Start a sealed layer from an empty ring and far field ("cortiq-engine
 * 0.8.51 src/gpu_wgpu/o1_batch.rs", struct State and the meta layout of
 * o1b_meta; an empty far field has M = -inf, Z = 0 as o1b_far_e's comment
 * states).
 *   state          device, o1_state_bytes(geom) bytes, 256-byte aligned; overwritten
 *   group_windows  host [G] or NULL: each group's window (meta slot 3),
 *                  0 = geom->window; every value <= geom->window
 *   sink_k, sink_v device [G][ns][d], [G][ns][dv] (may be NULL if ns == 0)
 *   k_tilde        device [G][m][d]      landmark keys, one set per group
 *   q_tilde        device [G][hpg][m][d] landmark queries, per head
 *   mu             device [G*hpg][m][m]  mu[a][b], a = landmark key, b = query
 *   pos0           absolute position of the first row (rotation angle)
 * Sinks and landmarks are used as given (already rotated). Asynchronous. */
O1_API int o1_state_init(void *state, const o1_geom *geom, const int32_t *group_windows,
                  const float *sink_k, const float *sink_v, const float *k_tilde,
                  const float *q_tilde, const float *mu, int64_t pos0, void *stream);

/* Attention of `rows` consecutive rows, and the state advanced past them
 * ("cortiq-engine 0.8.51 src/gpu_wgpu/o1_batch.rs": encode and the kernels
 * o1b_far_e, o1b_attend, o1b_far_commit, o1b_ring_commit, o1b_meta; gate as
 * dory_gate1 of "cortiq-engine 0.8.77 src/gpu_wgpu/dory.rs").
 *   q     device [rows][G*hpg][d]  queries, NOT rotated (rotated here at pos)
 *   k     device [rows][G][d]      keys, not rotated
 *   v     device [rows][G][dv]
 *   gate  device [rows][G*hpg][dv] gate logits, or NULL for no gate
 *   out   device [rows][G*hpg][dv] o / (1 + exp(-gate)); must not alias q/k/v/gate
 *   scratch, scratch_bytes  device scratch, at least o1_scratch_bytes(geom, 1)
 * The output equals the rows processed one at a time (rope, far insert, ring
 * push, attend, gate), up to rounding. Asynchronous.
 * Window path: when d % 64 == 0, d <= 256, dv % 32 == 0, dv <= 256 and
 * window >= 512, the window part of a pass with two or more rows runs on the
 * tensor cores, each fp32 operand split into two fp16 halves (hi + lo, three
 * products). It needs every rotated query, rotated key and value to lie
 * inside the fp16 range (|x| < 65504); one outside it raises
 * O1_FLAG_FP16_RANGE in the state's flags and that pass's output is not
 * valid. Other geometries, and one-row calls (which take the one-row path),
 * run in fp32 throughout. */
O1_API int o1_chunk_attend(void *state, const o1_geom *geom, void *scratch, size_t scratch_bytes,
                    const float *q, const float *k, const float *v, const float *gate,
                    int32_t rows, float *out, void *stream);

/* Speculative verification ("cortiq-engine 0.8.82 src/gpu_metal/o1c.rs":
 * encode with commit = false, then spec_commit over the accepted rows).
 *
 * o1_chunk_attend_spec: the attention of `rows` draft rows, exactly as
 * o1_chunk_attend would compute it (same arguments, layouts, checks and
 * output), but the state is left as it was: no far insert, ring push, meta
 * or position change. The draft must fit in one pass of the scratch
 * (rows <= the max_rows the scratch was sized for), else O1_ERR_ARG. A
 * one-row draft runs as a one-row pass of the chunk path, not the decode
 * path. Asynchronous.
 *
 * o1_spec_commit: moves the state over the first `rows` accepted rows, given
 * their keys and values again (k [rows][G][d] unrotated, v [rows][G][dv],
 * device, 16-byte aligned; the same values the verify call was given): the
 * rotation of the keys at the state's position, the far insert of every key
 * they evict, the ring push, meta and position. The state afterwards equals
 * the one o1_chunk_attend over those rows leaves, up to rounding; nothing is
 * attended and no output is written. rows = 0 does nothing. Rows above the
 * scratch's capacity run as several passes. Same scratch rules as
 * o1_chunk_attend. Asynchronous. */
O1_API int o1_chunk_attend_spec(void *state, const o1_geom *geom, void *scratch, size_t scratch_bytes,
                                const float *q, const float *k, const float *v, const float *gate,
                                int32_t rows, float *out, void *stream);
O1_API int o1_spec_commit(void *state, const o1_geom *geom, void *scratch, size_t scratch_bytes,
                          const float *k, const float *v, int32_t rows, void *stream);

/* Exact sliding-window attention, the comparator of the sealed layer (the
 * pages time the same model chunk with exact attention against the sealed
 * layer's per-row loop; "cortiq-engine 0.8.77 src/gpu_wgpu/dory.rs",
 * dory_score / dory_soft / dory_sum / dory_gate). Each row attends to the
 * sinks and to the last min(group window, len + r + 1) keys of [ring, oldest
 * first] ++ [this call's rows] ending at its own; keys that leave the window
 * are dropped, and there is no far field. Same arguments, layouts, checks,
 * rotation and gate as o1_chunk_attend, and the same window kernels. The
 * state is only read (no push, no position change), so the rows must fit in
 * one pass of the scratch, else O1_ERR_ARG. From a fresh state with a window
 * of at least `rows`, the output is exact causal softmax attention over the
 * sinks and every key. Asynchronous. */
O1_API int o1_window_attend(void *state, const o1_geom *geom, void *scratch, size_t scratch_bytes,
                            const float *q, const float *k, const float *v, const float *gate,
                            int32_t rows, float *out, void *stream);

/* One row (a decode step): the same as o1_chunk_attend with rows = 1, by a
 * path built for it ("cortiq-engine 0.8.82 src/gpu_metal/o1c.rs" encode_tok:
 * near partials split across blocks, the far part, a merge, the commit).
 *   q [G*hpg][d], k [G][d], v [G][dv], gate [G*hpg][dv] or NULL, out [G*hpg][dv]
 *   scratch  device, at least o1_scratch_bytes(geom, 1) bytes
 * Where that path's shared memory would exceed a block's (windows of a few
 * hundred thousand keys and more), the row runs as a one-row chunk pass,
 * with the same result. Asynchronous. */
O1_API int o1_token_attend(void *state, const o1_geom *geom, void *scratch, size_t scratch_bytes,
                    const float *q, const float *k, const float *v, const float *gate,
                    float *out, void *stream);

/* Stages of one chunk pass, in launch order: rope, far_block, far_tscan,
 * side_readout, gather_tc, near, merge, commit. The far-field stages
 * (far_block .. side_readout) run on a second, high-priority stream of the
 * library's, concurrently with gather_tc and near; it is forked from and
 * joined back into the caller's stream by events, so a stream capture of a
 * call captures both branches. The stream and its two events are created by
 * the first call on each host thread and device (make that call before a
 * stream capture) and live until that thread exits. A stage that does not apply to the geometry
 * (the fp16 panel gather outside the tensor-core window path) launches
 * nothing and times as empty. A pass of at most 16 rows runs its far field
 * and sinks as one short kernel (timed as side_readout; far_block and
 * far_tscan stay empty) and, from 2 rows, its window as key-slice kernels
 * (timed as near). */
#define O1_NUM_STAGES 8

/* o1_chunk_attend that also records caller-created CUDA events (cudaEvent_t
 * handles, passed as void*): events[2i] just before and events[2i + 1] just
 * after stage i of a pass, on the stream that stage runs on, so that
 * cudaEventElapsedTime(events[2i], events[2i + 1]) is stage i's time (with
 * the other branch running concurrently). With several passes (rows above
 * the scratch's capacity) the events end up holding the last pass. n_events
 * must be at least 2 * O1_NUM_STAGES. Same arguments, checks and result as
 * o1_chunk_attend otherwise. */
O1_API int o1_chunk_attend_timed(void *state, const o1_geom *geom, void *scratch, size_t scratch_bytes,
                                 const float *q, const float *k, const float *v, const float *gate,
                                 int32_t rows, float *out, void *const *events, int32_t n_events,
                                 void *stream);

/* Name of stage i of a chunk pass (NULL outside [0, O1_NUM_STAGES)). The
 * pages time a forward stage by stage by keeping only some dispatch kinds
 * ("cortiq-engine 0.8.77 src/gpu_wgpu/dory.rs", the keep-one stage table);
 * here each stage records events around itself instead, and every stage
 * still runs. */
O1_API const char *o1_stage_name(int32_t stage);

/* Size of the library's own device scratch used by o1_token_attend_noalloc:
 * 4 MiB, held by every GPU that loads the library until the process exits. */
#define O1_NOALLOC_SCRATCH_BYTES (4u << 20)

/* o1_token_attend for callers that cannot allocate device memory: no
 * scratch argument, no cudaMalloc, cudaFree or allocating library call.
 * For a plugin whose interface hands over no workspace, or a decode loop
 * that must not call cudaMalloc (it can synchronise the device and stall
 * other streams) nor keep a buffer of its own. The paper has no
 * counterpart; this is a convenience of this library.
 *   q, k, v, gate, out, state, stream: as o1_token_attend.
 * The scratch is one static device array of O1_NOALLOC_SCRATCH_BYTES in
 * this library, shared by every call on a device: calls that overlap on
 * the GPU (other streams, other threads) race on it, so serialise them.
 * Nothing in it needs to start at zero: a call writes every scratch value
 * before reading it. The first call on each device looks the array's
 * device address up (cudaGetSymbolAddress, that device current) and keeps
 * it for the life of the process; make that first call before any stream
 * capture. The kept address does not survive cudaDeviceReset of that device
 * (a new context holds the array elsewhere): do not reset a device and go on
 * calling this entry point on it in the same process. Returns O1_ERR_UNSUPPORTED when the
 * geometry's one-row scratch exceeds O1_NOALLOC_SCRATCH_BYTES, else as
 * o1_token_attend. */
O1_API int o1_token_attend_noalloc(void *state, const o1_geom *geom, const float *q, const float *k,
                                   const float *v, const float *gate, float *out, void *stream);

/* Copy the state's mutable parts to host memory (NULL fields skipped).
 * Synchronises `stream`. Returns O1_ERR_STATE if the state's header does not
 * hold this geometry.
 * What is read is the state a chunk leaves behind for the next chunk or the
 * one-row path to carry on from ("cortiq-engine 0.8.51
 * src/gpu_wgpu/o1_batch.rs", module doc on o1b_far_commit, o1b_ring_commit
 * and o1b_meta; the buffers of struct State): meta, ring keys and values by
 * slot, and the far field M, Z, T. */
O1_API int o1_state_read(const void *state, const o1_geom *geom, o1_state_host *dst, void *stream);

/* Overwrite the state's mutable parts from host memory (NULL fields kept):
 * snapshots and test set-up. Synchronises `stream`. The caller keeps the
 * state consistent (len <= group window, head < group window, M = -inf
 * exactly where farl == 0, ...).
 * The same parts as o1_state_read: the state a chunk hands on to the next
 * chunk or to the one-row path ("cortiq-engine 0.8.51
 * src/gpu_wgpu/o1_batch.rs", module doc and struct State). The pages upload
 * a sealed layer's state from the host the same way ("cortiq-engine 0.8.77
 * src/gpu_wgpu/dory.rs", seal: the far states built on the CPU are
 * uploaded). */
O1_API int o1_state_write(void *state, const o1_geom *geom, const o1_state_host *src, void *stream);

/* Sticky conditions a kernel records in the state header (bits of the value
 * o1_state_flags returns). */
#define O1_FLAG_WAIT_EXPIRED 1u  /* a bounded in-kernel wait ran out (about 2 s);
                                    that pass's output is incomplete      */
#define O1_FLAG_FP16_RANGE 2u    /* an operand of the tensor-core window path
                                    was outside the fp16 range             */
#define O1_FLAG_BACK_REFUSED 4u  /* an o1_state_back was larger than some
                                    group could rewind; nothing was changed */

/* Rewind the last `rows` ring pushes of every KV group, for looped-layer KV
 * modes that push the same positions again ("cortiq-engine 0.8.77
 * src/gpu_wgpu/dory.rs", dory_o1_back, applied once per row): a full ring
 * (len == group window) steps its head back by one and forgets one eviction
 * (farl - 1) per row; a ring not yet full drops its newest entry (len - 1).
 * The position moves back by `rows`. Ring contents and the far field (M, Z,
 * T) are not undone, as on the page: keys already folded into the far field
 * stay there. A rewind some group cannot take in full (len < rows while not
 * full, farl < rows while full) or one longer than the position is refused on
 * the device, with nothing changed, and raises O1_FLAG_BACK_REFUSED (the
 * state's meta lives on the device, so this call cannot see it). rows = 0
 * does nothing. One single-thread launch; asynchronous. */
O1_API int o1_state_back(void *state, const o1_geom *geom, int32_t rows, void *stream);

/* Limit, in SM clock cycles, of the kernels' waits (on their own copies and
 * tensor-core work) for calls made from now on, in this process; a call
 * captured in a CUDA graph keeps the limit it was captured with.
 * cycles < 1, or above the default of 4e9 (about 2 s at the maximum SM
 * clock), restores the default. A wait that runs out raises
 * O1_FLAG_WAIT_EXPIRED and that call's output is not valid; the kernel still
 * waits, with the default limit, for the work it had already issued before
 * it exits. A tiny limit makes the first waits run out on purpose, which is
 * how that path is tested; in use the default is meant to stay. Host-only,
 * no CUDA call; always O1_OK. (The pages' kernels wait on no barrier of
 * this kind, so there is no counterpart to cite.) */
O1_API int o1_set_wait_limit(int64_t cycles);

/* Read the state's flags into *flags (host) and, if `clear` is non-zero,
 * reset them to 0. Synchronises `stream`.
 * The pages report a failed dispatch or readback through the encoder's
 * boolean result ("cortiq-engine 0.8.82 src/gpu_metal/o1c.rs", encode and
 * spec_commit return false; the command buffer's error status is checked).
 * A kernel here cannot return a value, so it records such conditions as
 * these sticky bits. */
O1_API int o1_state_flags(void *state, const o1_geom *geom, uint32_t *flags, int32_t clear, void *stream);

/* A static, human-readable name for a status code. (The pages' geometry
 * gates refuse a shape instead of running it: "cortiq-engine 0.8.82
 * src/gpu_metal/o1c.rs", admits and tok_ok; this library returns
 * O1_ERR_UNSUPPORTED there.) */
O1_API const char *o1_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* O1_H */
