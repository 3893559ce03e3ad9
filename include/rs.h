/*
 * rs.h - C ABI of librs, a single-GPU library for the ReplaySSM decode path
 * (Mamba-2 and Gated DeltaNet layers) with hand-written sm_103a kernels.
 *
 * Sources, cited on every declaration by a "Source:" line:
 *   [CSI]  "ReplaySSM: Cache SSM Inputs, Not State" (a summary page): sections
 *          "What it claims", "How it works" (its bullets and flowchart),
 *          "Evidence" and "Limits";
 *   [THR]  "Songlin Yang releases ReplaySSM, cutting hybrid SSM memory
 *          traffic in half to enable 2x faster speculative decoding" (the
 *          author's thread): posts [2/N] to [6/N] and the replies under them;
 *   [TLDR] "ReplaySSM speeds up SSM decoding and runs in production in
 *          GLM-5.3-Flash and Kimi-K3": its TLDR;
 *   [ABS]  the ReplaySSM paper abstract.
 * "Source: none" marks library plumbing that has no counterpart there.
 *
 * The method ([CSI] "How it works"; [ABS]) keeps each sequence's
 * recurrent state S (P x N per head) as
 *
 *     a checkpoint S_c  +  a circular buffer of the SSM inputs since S_c,
 *
 * so that after h buffered records S = gamma * S_c + sum_j w_j v_j k_j^T,
 * with w_j the product of the decays after record j and gamma the product of
 * all of them.  A decode step appends its record and computes its output
 * straight from that form, without writing the state back; a new checkpoint
 * is stored once per window, when L records have been buffered (a "flush").
 * Speculative verification appends T draft records and computes all T
 * outputs from one checkpoint read; accepting a prefix or rolling back only
 * moves pointers.
 *
 * ---------------------------------------------------------------- conventions
 * Ownership: the caller allocates every buffer (device memory unless stated)
 *   and passes raw pointers; rs_state_bytes_for() gives the sizes.  The library
 *   allocates nothing and keeps no per-layer state.  All pointers to device
 *   arrays must be 16-byte aligned.
 * State kept between calls: only per-device launch facts, each set once per
 *   device under a lock: every kernel's dynamic shared-memory opt-in and the
 *   device's attributes (SM count, shared-memory limits); plus the static
 *   counters of rs_decode_mamba2_noalloc.
 * Streams: every call that touches the GPU takes a stream (a cudaStream_t,
 *   passed as void*; NULL = legacy default stream) and only enqueues work on
 *   it, except rs_get_status, which synchronises that stream.
 * Devices and threads: a call runs on the calling thread's current device
 *   (device ordinals below 64).  A process may drive several devices, and
 *   several host threads may call at once, on different layers or streams.
 * Errors: every call returns rs_status and never aborts.  Argument problems
 *   found on the host return RS_ERR_INVALID_ARG / RS_ERR_UNSUPPORTED before
 *   anything is enqueued.  A failed launch returns RS_ERR_CUDA.  Problems only
 *   visible on the device (a pointer state that breaks a rule below) set bits
 *   of the device status word, which rs_get_status reads; kernels never trap.
 * Types: "bf16" arrays are passed as raw 16-bit patterns (uint16_t); fp32 is
 *   float.  Outputs y are fp32.
 *
 * Layouts (row-major, innermost last):
 *   checkpoint (both precisions)  [B][H][N][P]   key index n, then value index p
 *   Mamba-2 step inputs  x [B][T][H][P] bf16, dt [B][T][H] f32,
 *                        Bm, Cm [B][T][G][N] bf16, A [H] f32, D [H] f32
 *   GDN step inputs      q, k [B][T][G][N] bf16 (k-heads), v [B][T][H][P] bf16,
 *                        alpha, beta [B][T][H] f32
 *   KDA step inputs      as GDN, but alpha [B][T][H][N] f32 (one decay per key channel)
 *   outputs              y [B][T][H][P] f32
 *   (T = 1 for the decode calls; the T axis may then be left out.)
 *   Mamba-2 head h uses B/C group h / (H/G); GDN (and KDA) v-head h uses k-head h / (H/G).
 */
#ifndef RS_H
#define RS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    RS_OK = 0,
    RS_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad size or count   */
    RS_ERR_UNSUPPORTED = 2,  /* shape or mode without a kernel instantiation */
    RS_ERR_CAPACITY = 3,     /* capacity below max(L, T_max) + T_max         */
    RS_ERR_CUDA = 4,         /* a CUDA call failed (launch or copy)          */
    RS_ERR_DEVICE = 5,       /* the device status word has bits set          */
    RS_ERR_STATIC_LIMIT = 6  /* B above RS_STATIC_MAX_SEQS (rs_decode_mamba2_noalloc) */
} rs_status;

/* Bits of the device status word. */
#define RS_DEV_CAPACITY 0x1u       /* records would overflow the circular buffer; sequence skipped */
#define RS_DEV_ACCEPT 0x2u         /* accepted length outside 0..nd; clamped                     */
#define RS_DEV_DRAFTS_PENDING 0x4u /* decode/verify/append with uncommitted drafts; drafts dropped */
#define RS_DEV_TIMEOUT 0x8u        /* an in-kernel wait gave up after its time limit; results invalid */

/* RS_KDA: Gated DeltaNet with one decay per key channel, alpha_t in R^N
 * (a reading of Kimi Delta Attention, which [CSI] "Limits" names as
 * compatible without defining it): D_t = S_{t-1} diag(alpha_t),
 * u_t = beta_t (v_t - D_t k_t), S_t = D_t + u_t k_t^T, y_t = S_t q_t. */
typedef enum { RS_MAMBA2 = 0, RS_GDN = 1, RS_KDA = 2 } rs_kind;

/* Flag OR-ed into rs_layer_desc.precision: Gated DeltaNet records keep the
 * correction term u in bf16 (round to nearest even) instead of fp32, halving
 * the records' value bytes.  Outputs and folds then read rounded u: their
 * error bound is that of values read from bf16 (a measured variant; the
 * pages are silent on the buffer's precision).  RS_GDN only.
 * Source: [CSI] "How it works", Gated DeltaNet bullet (records store u). */
#define RS_U_BF16 0x10

typedef enum {
    RS_PREC_FP32 = 0,        /* fp32 checkpoint only                                          */
    RS_PREC_TWO = 1,         /* fp32 high-precision copy + bf16 low-precision copy: non-flush
                                steps read bf16, flushes read fp32 and write both             */
    RS_PREC_SHARED_BF16 = 2  /* one bf16 checkpoint serves reads and updates                  */
} rs_precision;

/* Shape of one layer.  Supported (P, N): Mamba-2 (64,128), (64,64);
 * GDN and KDA (128,128), (64,64); KDA with the fp32 checkpoint only.  1 <= B <= 65535, B * H <= 2^26 (more state than
 * a GPU holds; kernels index slabs with 32-bit integers), L >= 1, T_max in 0..8, and
 * max(L, T_max) + T_max <= capacity <= 32: a round of T drafts writes after
 * the h committed records it may fold, and h reaches L (or T_max, when
 * T_max > L, after a fully accepted round that folded). */
typedef struct {
    int32_t kind;      /* rs_kind                                              */
    int32_t B;         /* sequences                                            */
    int32_t H;         /* Mamba-2 heads / GDN value heads                      */
    int32_t G;         /* Mamba-2 B/C groups / GDN key heads; H % G == 0       */
    int32_t P;         /* Mamba-2 headdim / GDN d_v                            */
    int32_t N;         /* Mamba-2 dstate / GDN d_k                             */
    int32_t L;         /* window: a standard step flushes when it makes h >= L */
    int32_t T_max;     /* largest draft count of rs_verify (0: standard only)  */
    int32_t capacity;  /* circular buffer slots per sequence                   */
    int32_t precision; /* rs_precision, optionally | RS_U_BF16 (GDN)          */
} rs_layer_desc;

/* Per-layer state; every member is a caller-allocated device array. */
typedef struct {
    float *ckpt_hp;    /* fp32 checkpoint [B][H][N][P]; NULL for RS_PREC_SHARED_BF16 */
    uint16_t *ckpt_lp; /* bf16 checkpoint [B][H][N][P]; NULL for RS_PREC_FP32        */
    void *buf_v;       /* records' values: Mamba-2 x bf16 [B][cap][H][P];
                          GDN / KDA correction term u fp32 [B][cap][H][P]
                          (bf16 with RS_U_BF16)                                       */
    uint16_t *buf_k;   /* records' keys (Mamba-2 B / GDN k) bf16 [B][cap][G][N]       */
    float *buf_a;      /* records' decays alpha, fp32 [B][cap][H] (Mamba-2: exp(dt A));
                          KDA [B][cap][H][N]                                          */
    float *buf_s;      /* Mamba-2 records' dt, fp32 [B][cap][H] (v = dt x); NULL otherwise */
    int32_t *base;     /* [B] slot of the first record after the checkpoint          */
    int32_t *h;        /* [B] committed records after the checkpoint                 */
    int32_t *nd;       /* [B] appended, not yet accepted draft records               */
    uint32_t *arrive;  /* [B + 2] per-sequence arrival counters and the launch's two
                          unit-scheduling counters (kernel scratch; rs_init clears it) */
    uint32_t *status;  /* [1] device status word (RS_DEV_* bits)                     */
} rs_state;

/* Byte sizes of the rs_state arrays for a descriptor (0 for an unused array). */
typedef struct {
    size_t ckpt_hp, ckpt_lp, buf_v, buf_k, buf_a, buf_s, base, h, nd, arrive, status;
} rs_state_bytes;

/* Inputs of several records per sequence, [B][n][...] as in the layouts above.
 * Members of the other family must be NULL. */
typedef struct {
    const uint16_t *x;  const float *dt; const float *A;
    const uint16_t *Bm; const uint16_t *Cm; const float *D; /* D may be NULL (= 0) */
    const uint16_t *q;  const uint16_t *k;  const uint16_t *v;
    const float *alpha; const float *beta;
} rs_inputs;

/* ------------------------------------------------------------------- host-only */
/* Text of a status code.  Source: none (library plumbing). */
const char *rs_status_string(rs_status s);
/* Library name, version and target architecture.  Source: none (library plumbing). */
const char *rs_version(void);
/* Name and text of the CUDA error behind the calling thread's most recent
 * RS_ERR_CUDA ("" if none); for diagnostics.  Source: none (library plumbing). */
const char *rs_last_cuda_error(void);

/* Validates the descriptor and fills the byte sizes of the arrays of the
 * per-layer state: the checkpoint in one or two precisions, the circular
 * buffer of records (values, keys, decays), and the per-sequence pointers.
 * Host only; out must not be NULL.
 * Source: [CSI] "How it works", standard-decoding bullet (a checkpoint plus a
 * buffer of the steps' (alpha, v, k) records), speculative bullet (a circular
 * buffer of capacity L + T) and "Two precisions" bullet; [CSI] "What it
 * claims" (an FP32 state of 4 MiB per sequence and layer). */
rs_status rs_state_bytes_for(const rs_layer_desc *desc, rs_state_bytes *out);

/* ---------------------------------------------------------------- state setup */
/* Writes the checkpoint from init (fp32 [B][H][N][P], device; NULL = zeros):
 * the fp32 copy and/or its bf16 rounding (nearest-even) per the precision
 * mode.  Clears base, h, nd, the arrival counters and the status word.
 * This is the two-precision checkpoint writer on its own.
 * Source: [CSI] "How it works", "Two precisions" bullet. */
rs_status rs_init(const rs_layer_desc *desc, const rs_state *st, const float *init, void *stream);

/* Reads the device status word into *bits (host), after synchronising the
 * stream; clears it if clear != 0.  Returns RS_ERR_DEVICE if any bit was set.
 * Source: none (library plumbing: how device-side problems reach the host). */
rs_status rs_get_status(const rs_state *st, uint32_t *bits, int clear, void *stream);

/* ------------------------------------------------------------ standard decode */
/* One Mamba-2 decode step for all B sequences.  Per sequence: append the
 * record (x_t, dt_t, B_t) and write y_t = gamma S_c C_t + sum_j w_j dt_j x_j
 * (B_j . C_t) + D x_t without writing the state.  When the record makes
 * h >= L the same launch folds all h records into the checkpoint,
 * S_c <- gamma S_c + V diag(w) K^T (the flush route), and resets h to 0.
 * alpha_t = exp(dt_t A_h).  Drafts pending are dropped (RS_DEV_DRAFTS_PENDING).
 * Source: [CSI] "How it works", standard-decoding bullet; [THR] posts [4/N]
 * and [5/N] (append instead of writing the state; the output straight from
 * the buffer) and the replies on the flush route (the new state as one
 * product V K^T, the output from it). */
rs_status rs_decode_mamba2(const rs_layer_desc *desc, const rs_state *st, const uint16_t *x,
                           const float *dt, const float *A, const uint16_t *Bm,
                           const uint16_t *Cm, const float *D, float *y, void *stream);

/* One Gated DeltaNet decode step: u_t = beta_t (v_t - alpha_t S_{t-1} k_t)
 * where S_{t-1} k_t is itself replayed from the checkpoint and the buffered
 * u_j; the record stores u_t in place of v_t; y_t = S_t q_t.  One checkpoint
 * read serves both S k and S q.  Flush rule as for rs_decode_mamba2.
 * Source: [CSI] "How it works", Gated DeltaNet bullet. */
rs_status rs_decode_gdn(const rs_layer_desc *desc, const rs_state *st, const uint16_t *q,
                        const uint16_t *k, const uint16_t *v, const float *alpha,
                        const float *beta, float *y, void *stream);

/* One decode step of a layer with per-channel decays (RS_KDA): as
 * rs_decode_gdn, with alpha fp32 [B][H][N].  In replay form the decay
 * weights become vectors over the key channels: y_t = S_c (gamma(t) (.) q_t)
 * + sum_j u_j ((w_j(t) (.) k_j) . q_t), and the flush writes
 * S_c <- S_c diag(gamma) + sum_j u_j (w_j (.) k_j)^T.  Records keep the
 * decay vectors (fp32 [B][cap][H][N]).
 * Source: [CSI] "Limits" (Kimi Delta Attention named as compatible but not
 * implemented) and "How it works", Gated DeltaNet bullet. */
rs_status rs_decode_kda(const rs_layer_desc *desc, const rs_state *st, const uint16_t *q,
                        const uint16_t *k, const uint16_t *v, const float *alpha,
                        const float *beta, float *y, void *stream);

/* ------------------------------------------------------------------ speculative */
/* Speculative verification of T drafts (1 <= T <= T_max), either family.
 * Appends the T draft records and writes all T outputs y [B][T][H][P] from one
 * checkpoint read and the buffer.  Per sequence, if h + T > L the committed
 * records (never the drafts) are folded into the checkpoint in the same
 * launch (reading the fp32 copy and writing both copies in two-precision
 * mode); otherwise the low-precision copy is read in two-precision mode.
 * Sets nd = T.
 * Source: [CSI] "How it works", speculative bullet and flowchart; [THR] post
 * [5/N] (the output-only form turns draft verification into GEMMs). */
rs_status rs_verify(const rs_layer_desc *desc, const rs_state *st, int T, const rs_inputs *in,
                    float *y, void *stream);

/* Accepts a prefix of the drafts: h += accepted[b], nd = 0 (a pointer move).
 * accepted: device int32 [B], each in 0..nd (else clamped, RS_DEV_ACCEPT).
 * Source: [CSI] "How it works", the flowchart's last step (advance the
 * pointer by the accepted length) and speculative bullet; [TLDR] (rolling
 * back a wrong guess is just a pointer move). */
rs_status rs_commit(const rs_layer_desc *desc, const rs_state *st, const int32_t *accepted,
                    void *stream);

/* Discards the drafts: nd = 0.  Their records are overwritten later.
 * Source: [THR] post [4/N] (rollback becomes a pointer move); [CSI] "How it
 * works", speculative bullet (rejected records are simply overwritten). */
rs_status rs_rollback(const rs_layer_desc *desc, const rs_state *st, void *stream);

/* ---------------------------------------------------------------- maintenance */
/* Appends n committed Mamba-2 records per sequence without computing outputs
 * or flushing (x, dt, Bm of in, each [B][n][...]).  Needs nd == 0 and
 * h + n <= capacity per sequence (else that sequence is skipped and a status
 * bit set).  GDN records depend on the state, so GDN returns RS_ERR_UNSUPPORTED.
 * Source: [CSI] "How it works", standard-decoding bullet (each step appends
 * the token's inputs to a buffer); [THR] post [4/N]. */
rs_status rs_append(const rs_layer_desc *desc, const rs_state *st, int n, const rs_inputs *in,
                    void *stream);

/* Folds every committed record into the checkpoint now (h -> 0), writing
 * both copies in two-precision mode.  Drafts stay appended.
 * Source: [CSI] "How it works", standard-decoding bullet (the checkpoint
 * written when the window fills) and speculative bullet (flushes fold only
 * committed records, so they may run at any time); [THR] the reply on prefix
 * caching (a cached state must not be stale). */
rs_status rs_flush(const rs_layer_desc *desc, const rs_state *st, void *stream);

/* Writes the committed state S = gamma S_c + sum_{j<h} w_j v_j k_j^T to out
 * (fp32 [B][H][N][P], device) without changing anything; an export of the
 * current state, e.g. for prefix caching.
 * Source: [CSI] "How it works", standard-decoding bullet (the state rebuilt
 * as the decayed checkpoint plus a sum over the buffered inputs); [THR] the
 * reply on prefix caching. */
rs_status rs_materialize(const rs_layer_desc *desc, const rs_state *st, float *out, void *stream);

/* ---------------------------------------------------------- eager baselines */
/* Conventional decode that loads and stores the state every step:
 * S <- alpha S + v k^T, y = S q (+ D x).  S: fp32 [B][H][N][P], updated in
 * place.  The computation uses kind, B, H, G, P, N of desc (T_max too for the
 * snapshot calls); the whole descriptor must still pass the usual validation.
 * Source: [THR] post [2/N] (loading and storing the state every step); [ABS]
 * (eager state management); the GDN form as in [CSI] "How it works", Gated
 * DeltaNet bullet. */
rs_status rs_eager_step_mamba2(const rs_layer_desc *desc, float *S, const uint16_t *x,
                               const float *dt, const float *A, const uint16_t *Bm,
                               const uint16_t *Cm, const float *D, float *y, void *stream);
rs_status rs_eager_step_gdn(const rs_layer_desc *desc, float *S, const uint16_t *q,
                            const uint16_t *k, const uint16_t *v, const float *alpha,
                            const float *beta, float *y, void *stream);
/* The eager step with per-channel decays (alpha fp32 [B][H][N]):
 * S <- S diag(alpha) + u k^T with u = beta (v - S diag(alpha) k), y = S q.
 * Source: [THR] post [2/N] (loading and storing the state every step); the
 * per-channel decay as read for rs_decode_kda from [CSI] "Limits". */
rs_status rs_eager_step_kda(const rs_layer_desc *desc, float *S, const uint16_t *q,
                            const uint16_t *k, const uint16_t *v, const float *alpha,
                            const float *beta, float *y, void *stream);

/* Per-draft snapshot baseline for speculative decoding: one state kept per
 * draft token.  pool: fp32 [B][T_max+1][H][N][P];
 * cur: device int32 [B], the pool slot holding each sequence's committed state.
 * Reads slot cur[b], runs the eager recurrence over the T drafts, writes each
 * intermediate state to slot (cur[b] + 1 + i) % (T_max + 1) and the outputs to
 * y [B][T][H][P].
 * Source: [THR] post [3/N] (a separate state for every draft token);
 * [CSI] "Evidence" (vLLM's per-draft snapshots as the comparison). */
rs_status rs_eager_verify_snapshots(const rs_layer_desc *desc, float *pool, const int32_t *cur,
                                    int T, const rs_inputs *in, float *y, void *stream);

/* Selects the snapshot of the accepted prefix: cur[b] = (cur[b] +
 * accepted[b]) % (T_max + 1).  status (device [1], may be NULL) gets
 * RS_DEV_ACCEPT for an accepted length outside 0..T_max.
 * Source: [THR] post [3/N] (rolling back to the state kept for the last
 * accepted draft). */
rs_status rs_eager_select(const rs_layer_desc *desc, int32_t *cur, const int32_t *accepted,
                          uint32_t *status, void *stream);

/* ------------------------------------------------- decode without caller scratch */
/* Largest batch rs_decode_mamba2_noalloc accepts. */
#define RS_STATIC_MAX_SEQS 4096

/* rs_decode_mamba2 for callers that cannot give the library any device memory
 * beyond inputs, outputs and the layer state.  Examples are an engine plugin
 * that only receives pre-planned tensors, or a server that forbids device
 * allocation after start-up.  The per-sequence arrival counters, which
 * rs_decode_mamba2 keeps in st->arrive (that member is ignored here and may be
 * NULL), live in a static device array of this library instead (4096 counters
 * and the two unit-scheduling counters: 16 KiB + 8 bytes).
 *   - B <= RS_STATIC_MAX_SEQS, else RS_ERR_STATIC_LIMIT and nothing is enqueued.
 *   - The first call in a device context looks up the array's address with
 *     that device current; make it before any stream capture.  The address is
 *     tagged with the context's unique ID, so the first call in a new context
 *     of the device (after cudaDeviceReset, say) looks it up again and
 *     should come before any capture too.  Each call clears the counters it
 *     uses on `stream`, then runs the same kernel as rs_decode_mamba2 with the
 *     same results.
 *   - All calls share the array: calls that overlap on the GPU race, so
 *     serialise them.  The array stays allocated on every device that loaded
 *     the library until the process exits.
 *   - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 * Source: none (no counterpart in the paper: a packaging choice). */
rs_status rs_decode_mamba2_noalloc(const rs_layer_desc *desc, const rs_state *st, const uint16_t *x,
                                   const float *dt, const float *A, const uint16_t *Bm,
                                   const uint16_t *Cm, const float *D, float *y, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* RS_H */
