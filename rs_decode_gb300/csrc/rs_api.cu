// C-ABI entry points of librs: argument validation on the host, then one or
// two kernel launches on the caller's stream.  No entry point allocates
// memory; between calls the library keeps only per-device launch facts (the
// kernels' shared-memory opt-in and the device's attributes).
#include <stdint.h>
#include <stdio.h>

#include <cuda_runtime.h>

#include "rs.h"
#include "rs_common.cuh"
#include "rs_internal.h"

using namespace rs;

namespace {

constexpr long long kMaxSlabs = 1ll << 26;

inline bool aligned(const void *p, size_t a) { return p && (reinterpret_cast<uintptr_t>(p) % a) == 0; }

thread_local char g_last_cuda_error[160] = "";

}  // namespace

namespace rs {

rs_status check_desc(const rs_layer_desc *d) {
    if (!d) return RS_ERR_INVALID_ARG;
    if (d->kind != RS_MAMBA2 && d->kind != RS_GDN && d->kind != RS_KDA) return RS_ERR_INVALID_ARG;
    if (d->B < 1 || d->B > 65535 || d->H < 1 || d->G < 1 || d->H % d->G != 0) return RS_ERR_INVALID_ARG;
    // kernels index slabs (sequence x head) and units with 32-bit integers; 2^26
    // slabs of the smallest shape (64 x 64 bf16) are already 512 GiB
    if ((long long)d->B * d->H > kMaxSlabs) return RS_ERR_INVALID_ARG;
    if (d->P < 1 || d->N < 1 || d->L < 1 || d->T_max < 0 || d->T_max > kMaxT) return RS_ERR_INVALID_ARG;
    const int ckpt = d->precision & ~RS_U_BF16;
    if (ckpt < RS_PREC_FP32 || ckpt > RS_PREC_SHARED_BF16) return RS_ERR_INVALID_ARG;
    if (d->capacity > kMaxCap || d->capacity < 1) return RS_ERR_INVALID_ARG;
    // A standard step needs the h <= L - 1 records since the checkpoint plus
    // its own; a round of T drafts needs h + T, and after a fully accepted
    // round h can be max(L, T_max) (L when h + T <= L held, T_max after a
    // fold).  So max(L, T_max) + T_max slots always suffice, and some
    // sequence of calls needs all of them (L + T_max when T_max <= L).
    if (d->capacity < (d->L > d->T_max ? d->L : d->T_max) + d->T_max) return RS_ERR_CAPACITY;
    if (!replay_shape_supported(d->kind, d->P, d->N)) return RS_ERR_UNSUPPORTED;
    if (d->kind == RS_KDA && d->precision != RS_PREC_FP32) return RS_ERR_UNSUPPORTED;
    if ((d->precision & RS_U_BF16) && d->kind != RS_GDN) return RS_ERR_UNSUPPORTED;
    return RS_OK;
}

rs_status check_state(const rs_layer_desc *d, const rs_state *s, bool need_arrive) {
    if (!s) return RS_ERR_INVALID_ARG;
    const int ckpt = d->precision & ~RS_U_BF16;
    const bool need_hp = ckpt != RS_PREC_SHARED_BF16, need_lp = ckpt != RS_PREC_FP32;
    if (need_hp != (s->ckpt_hp != nullptr) || need_lp != (s->ckpt_lp != nullptr)) return RS_ERR_INVALID_ARG;
    if (need_hp && !aligned(s->ckpt_hp, 16)) return RS_ERR_INVALID_ARG;
    if (need_lp && !aligned(s->ckpt_lp, 16)) return RS_ERR_INVALID_ARG;
    if (!aligned(s->buf_v, 16) || !aligned(s->buf_k, 16) || !aligned(s->buf_a, 4)) return RS_ERR_INVALID_ARG;
    if ((d->kind == RS_MAMBA2) != (s->buf_s != nullptr)) return RS_ERR_INVALID_ARG;
    if (s->buf_s && !aligned(s->buf_s, 4)) return RS_ERR_INVALID_ARG;
    if (!aligned(s->base, 4) || !aligned(s->h, 4) || !aligned(s->nd, 4) || !aligned(s->status, 4))
        return RS_ERR_INVALID_ARG;
    if (need_arrive && !aligned(s->arrive, 4)) return RS_ERR_INVALID_ARG;
    return RS_OK;
}

rs_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return RS_OK;
    snprintf(g_last_cuda_error, sizeof g_last_cuda_error, "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
    return RS_ERR_CUDA;
}

// Inputs of one family; all other members must be null.
rs_status check_inputs(int kind, const rs_inputs *in, bool need_q) {
    if (!in) return RS_ERR_INVALID_ARG;
    if (kind == RS_MAMBA2) {
        if (!aligned(in->x, 16) || !aligned(in->dt, 4) || !aligned(in->A, 4) || !aligned(in->Bm, 16))
            return RS_ERR_INVALID_ARG;
        if (need_q && !aligned(in->Cm, 16)) return RS_ERR_INVALID_ARG;
        if (in->D && !aligned(in->D, 4)) return RS_ERR_INVALID_ARG;
        if (in->q || in->k || in->v || in->alpha || in->beta) return RS_ERR_INVALID_ARG;
    } else {
        // KDA reads its decay vectors 16 bytes at a time
        if (!aligned(in->q, 16) || !aligned(in->k, 16) || !aligned(in->v, 16) ||
            !aligned(in->alpha, kind == RS_KDA ? 16 : 4) || !aligned(in->beta, 4))
            return RS_ERR_INVALID_ARG;
        if (in->x || in->dt || in->A || in->Bm || in->Cm || in->D) return RS_ERR_INVALID_ARG;
    }
    return RS_OK;
}

}  // namespace rs

namespace {

ReplayParams replay_params(const rs_layer_desc *d, const rs_state *s, int mode, int T) {
    ReplayParams p = {};
    p.B = d->B; p.H = d->H; p.G = d->G; p.L = d->L; p.cap = d->capacity; p.T = T;
    p.prec = d->precision & ~RS_U_BF16; p.u16 = (d->precision & RS_U_BF16) != 0; p.mode = mode;
    p.ckpt_hp = s->ckpt_hp; p.ckpt_lp = s->ckpt_lp;
    p.buf_v = s->buf_v; p.buf_k = s->buf_k; p.buf_a = s->buf_a; p.buf_s = s->buf_s;
    p.base = s->base; p.h = s->h; p.nd = s->nd; p.arrive = s->arrive; p.status = s->status;
    return p;
}

void set_inputs(ReplayParams &p, const rs_inputs &in) {
    p.x = in.x; p.dt = in.dt; p.A = in.A; p.Bm = in.Bm; p.Cm = in.Cm; p.D = in.D;
    p.q = in.q; p.k = in.k; p.v = in.v; p.alpha = in.alpha; p.beta = in.beta;
}


#define RS_TRY(expr)                      \
    do {                                  \
        rs_status _s = (expr);            \
        if (_s != RS_OK) return _s;       \
    } while (0)

}  // namespace

extern "C" {

const char *rs_status_string(rs_status s) {
    switch (s) {
        case RS_OK: return "ok";
        case RS_ERR_INVALID_ARG: return "invalid argument";
        case RS_ERR_UNSUPPORTED: return "unsupported shape or mode";
        case RS_ERR_CAPACITY: return "buffer capacity below max(L, T_max) + T_max";
        case RS_ERR_CUDA: return "CUDA error";
        case RS_ERR_DEVICE: return "device status bits set";
        case RS_ERR_STATIC_LIMIT: return "batch above the static scratch limit (RS_STATIC_MAX_SEQS)";
    }
    return "unknown status";
}

const char *rs_version(void) { return "librs 0.1 (sm_103a)"; }

const char *rs_last_cuda_error(void) { return g_last_cuda_error; }

rs_status rs_state_bytes_for(const rs_layer_desc *d, rs_state_bytes *o) {
    RS_TRY(check_desc(d));
    if (!o) return RS_ERR_INVALID_ARG;
    const size_t B = d->B, H = d->H, G = d->G, P = d->P, N = d->N, C = d->capacity;
    const int ckpt = d->precision & ~RS_U_BF16;
    o->ckpt_hp = ckpt != RS_PREC_SHARED_BF16 ? B * H * N * P * 4 : 0;
    o->ckpt_lp = ckpt != RS_PREC_FP32 ? B * H * N * P * 2 : 0;
    o->buf_v = B * C * H * P * (d->kind == RS_MAMBA2 || (d->precision & RS_U_BF16) ? 2 : 4);
    o->buf_k = B * C * G * N * 2;
    o->buf_a = B * C * H * (d->kind == RS_KDA ? N : 1) * 4;
    o->buf_s = d->kind == RS_MAMBA2 ? B * C * H * 4 : 0;
    o->base = o->h = o->nd = B * 4;
    o->arrive = (B + 2) * 4;  // per-sequence arrival counters + the launch's two scheduling counters
    o->status = 4;
    return RS_OK;
}

rs_status rs_init(const rs_layer_desc *d, const rs_state *st, const float *init, void *stream) {
    RS_TRY(check_desc(d));
    RS_TRY(check_state(d, st));
    if (init && !aligned(init, 16)) return RS_ERR_INVALID_ARG;
    return cuda_status(init_launch(*d, *st, init, (cudaStream_t)stream));
}

rs_status rs_get_status(const rs_state *st, uint32_t *bits, int clear, void *stream) {
    if (!st || !aligned(st->status, 4) || !bits) return RS_ERR_INVALID_ARG;
    cudaStream_t s = (cudaStream_t)stream;
    uint32_t v = 0;
    if (cudaMemcpyAsync(&v, st->status, sizeof v, cudaMemcpyDeviceToHost, s) != cudaSuccess) return RS_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return RS_ERR_CUDA;
    if (clear) {
        if (cudaMemsetAsync(st->status, 0, sizeof v, s) != cudaSuccess) return RS_ERR_CUDA;
        if (cudaStreamSynchronize(s) != cudaSuccess) return RS_ERR_CUDA;
    }
    *bits = v;
    return v ? RS_ERR_DEVICE : RS_OK;
}

rs_status rs_decode_mamba2(const rs_layer_desc *d, const rs_state *st, const uint16_t *x, const float *dt,
                           const float *A, const uint16_t *Bm, const uint16_t *Cm, const float *D, float *y,
                           void *stream) {
    RS_TRY(check_desc(d));
    if (d->kind != RS_MAMBA2) return RS_ERR_INVALID_ARG;
    RS_TRY(check_state(d, st));
    rs_inputs in = {};
    in.x = x; in.dt = dt; in.A = A; in.Bm = Bm; in.Cm = Cm; in.D = D;
    RS_TRY(check_inputs(RS_MAMBA2, &in, true));
    if (!aligned(y, 16)) return RS_ERR_INVALID_ARG;
    ReplayParams p = replay_params(d, st, MODE_DECODE, 1);
    set_inputs(p, in);
    p.y = y;
    return cuda_status(replay_launch(p, d->kind, d->P, d->N, (cudaStream_t)stream));
}

rs_status rs_decode_gdn(const rs_layer_desc *d, const rs_state *st, const uint16_t *q, const uint16_t *k,
                        const uint16_t *v, const float *alpha, const float *beta, float *y, void *stream) {
    RS_TRY(check_desc(d));
    if (d->kind != RS_GDN) return RS_ERR_INVALID_ARG;
    RS_TRY(check_state(d, st));
    rs_inputs in = {};
    in.q = q; in.k = k; in.v = v; in.alpha = alpha; in.beta = beta;
    RS_TRY(check_inputs(RS_GDN, &in, true));
    if (!aligned(y, 16)) return RS_ERR_INVALID_ARG;
    ReplayParams p = replay_params(d, st, MODE_DECODE, 1);
    set_inputs(p, in);
    p.y = y;
    return cuda_status(replay_launch(p, d->kind, d->P, d->N, (cudaStream_t)stream));
}

rs_status rs_decode_kda(const rs_layer_desc *d, const rs_state *st, const uint16_t *q, const uint16_t *k,
                        const uint16_t *v, const float *alpha, const float *beta, float *y, void *stream) {
    RS_TRY(check_desc(d));
    if (d->kind != RS_KDA) return RS_ERR_INVALID_ARG;
    RS_TRY(check_state(d, st));
    rs_inputs in = {};
    in.q = q; in.k = k; in.v = v; in.alpha = alpha; in.beta = beta;
    RS_TRY(check_inputs(RS_KDA, &in, true));
    if (!aligned(y, 16)) return RS_ERR_INVALID_ARG;
    ReplayParams p = replay_params(d, st, MODE_DECODE, 1);
    set_inputs(p, in);
    p.y = y;
    return cuda_status(replay_launch(p, d->kind, d->P, d->N, (cudaStream_t)stream));
}

rs_status rs_verify(const rs_layer_desc *d, const rs_state *st, int T, const rs_inputs *in, float *y,
                    void *stream) {
    RS_TRY(check_desc(d));
    RS_TRY(check_state(d, st));
    if (T < 1 || T > d->T_max) return RS_ERR_INVALID_ARG;
    RS_TRY(check_inputs(d->kind, in, true));
    if (!aligned(y, 16)) return RS_ERR_INVALID_ARG;
    ReplayParams p = replay_params(d, st, MODE_VERIFY, T);
    set_inputs(p, *in);
    p.y = y;
    return cuda_status(replay_launch(p, d->kind, d->P, d->N, (cudaStream_t)stream));
}

rs_status rs_commit(const rs_layer_desc *d, const rs_state *st, const int32_t *accepted, void *stream) {
    RS_TRY(check_desc(d));
    RS_TRY(check_state(d, st));
    if (!aligned(accepted, 4)) return RS_ERR_INVALID_ARG;
    return cuda_status(commit_launch(d->B, accepted, st->h, st->nd, st->status, (cudaStream_t)stream));
}

rs_status rs_rollback(const rs_layer_desc *d, const rs_state *st, void *stream) {
    RS_TRY(check_desc(d));
    RS_TRY(check_state(d, st));
    return cuda_status(rollback_launch(d->B, st->nd, (cudaStream_t)stream));
}

rs_status rs_append(const rs_layer_desc *d, const rs_state *st, int n, const rs_inputs *in, void *stream) {
    RS_TRY(check_desc(d));
    if (d->kind != RS_MAMBA2) return RS_ERR_UNSUPPORTED;
    RS_TRY(check_state(d, st));
    if (n < 1 || n > d->capacity) return RS_ERR_INVALID_ARG;
    RS_TRY(check_inputs(RS_MAMBA2, in, false));
    return cuda_status(append_launch(*d, *st, n, *in, (cudaStream_t)stream));
}

rs_status rs_flush(const rs_layer_desc *d, const rs_state *st, void *stream) {
    RS_TRY(check_desc(d));
    RS_TRY(check_state(d, st));
    ReplayParams p = replay_params(d, st, MODE_FLUSH, 0);
    return cuda_status(replay_launch(p, d->kind, d->P, d->N, (cudaStream_t)stream));
}

rs_status rs_materialize(const rs_layer_desc *d, const rs_state *st, float *out, void *stream) {
    RS_TRY(check_desc(d));
    RS_TRY(check_state(d, st));
    if (!aligned(out, 16)) return RS_ERR_INVALID_ARG;
    ReplayParams p = replay_params(d, st, MODE_MATERIALIZE, 0);
    p.out = out;
    return cuda_status(replay_launch(p, d->kind, d->P, d->N, (cudaStream_t)stream));
}

rs_status rs_eager_step_mamba2(const rs_layer_desc *d, float *S, const uint16_t *x, const float *dt,
                               const float *A, const uint16_t *Bm, const uint16_t *Cm, const float *D, float *y,
                               void *stream) {
    RS_TRY(check_desc(d));
    if (d->kind != RS_MAMBA2) return RS_ERR_INVALID_ARG;
    if (!aligned(S, 16) || !aligned(y, 16)) return RS_ERR_INVALID_ARG;
    rs_inputs in = {};
    in.x = x; in.dt = dt; in.A = A; in.Bm = Bm; in.Cm = Cm; in.D = D;
    RS_TRY(check_inputs(RS_MAMBA2, &in, true));
    EagerParams p = {};
    p.B = d->B; p.H = d->H; p.G = d->G; p.T = 1; p.slots = 1; p.S = S;
    p.x = x; p.dt = dt; p.A = A; p.Bm = Bm; p.Cm = Cm; p.D = D; p.y = y;
    return cuda_status(eager_launch(p, d->kind, d->P, d->N, (cudaStream_t)stream));
}

rs_status rs_eager_step_gdn(const rs_layer_desc *d, float *S, const uint16_t *q, const uint16_t *k,
                            const uint16_t *v, const float *alpha, const float *beta, float *y, void *stream) {
    RS_TRY(check_desc(d));
    if (d->kind != RS_GDN) return RS_ERR_INVALID_ARG;
    if (!aligned(S, 16) || !aligned(y, 16)) return RS_ERR_INVALID_ARG;
    rs_inputs in = {};
    in.q = q; in.k = k; in.v = v; in.alpha = alpha; in.beta = beta;
    RS_TRY(check_inputs(RS_GDN, &in, true));
    EagerParams p = {};
    p.B = d->B; p.H = d->H; p.G = d->G; p.T = 1; p.slots = 1; p.S = S;
    p.q = q; p.k = k; p.v = v; p.alpha = alpha; p.beta = beta; p.y = y;
    return cuda_status(eager_launch(p, d->kind, d->P, d->N, (cudaStream_t)stream));
}

rs_status rs_eager_step_kda(const rs_layer_desc *d, float *S, const uint16_t *q, const uint16_t *k,
                            const uint16_t *v, const float *alpha, const float *beta, float *y, void *stream) {
    RS_TRY(check_desc(d));
    if (d->kind != RS_KDA) return RS_ERR_INVALID_ARG;
    if (!aligned(S, 16) || !aligned(y, 16)) return RS_ERR_INVALID_ARG;
    rs_inputs in = {};
    in.q = q; in.k = k; in.v = v; in.alpha = alpha; in.beta = beta;
    RS_TRY(check_inputs(RS_KDA, &in, true));
    EagerParams p = {};
    p.B = d->B; p.H = d->H; p.G = d->G; p.T = 1; p.slots = 1; p.S = S;
    p.q = q; p.k = k; p.v = v; p.alpha = alpha; p.beta = beta; p.y = y;
    return cuda_status(eager_launch(p, d->kind, d->P, d->N, (cudaStream_t)stream));
}

rs_status rs_eager_verify_snapshots(const rs_layer_desc *d, float *pool, const int32_t *cur, int T,
                                    const rs_inputs *in, float *y, void *stream) {
    RS_TRY(check_desc(d));
    if (T < 1 || T > d->T_max) return RS_ERR_INVALID_ARG;
    if (!aligned(pool, 16) || !aligned(cur, 4) || !aligned(y, 16)) return RS_ERR_INVALID_ARG;
    RS_TRY(check_inputs(d->kind, in, true));
    EagerParams p = {};
    p.B = d->B; p.H = d->H; p.G = d->G; p.T = T; p.slots = d->T_max + 1; p.S = pool; p.cur = cur;
    p.x = in->x; p.dt = in->dt; p.A = in->A; p.Bm = in->Bm; p.Cm = in->Cm; p.D = in->D;
    p.q = in->q; p.k = in->k; p.v = in->v; p.alpha = in->alpha; p.beta = in->beta; p.y = y;
    return cuda_status(eager_launch(p, d->kind, d->P, d->N, (cudaStream_t)stream));
}

rs_status rs_eager_select(const rs_layer_desc *d, int32_t *cur, const int32_t *accepted, uint32_t *status,
                          void *stream) {
    RS_TRY(check_desc(d));
    if (d->T_max < 1 || !aligned(cur, 4) || !aligned(accepted, 4)) return RS_ERR_INVALID_ARG;
    if (status && !aligned(status, 4)) return RS_ERR_INVALID_ARG;
    return cuda_status(select_launch(d->B, d->T_max + 1, cur, accepted, status, (cudaStream_t)stream));
}

}  // extern "C"
