// rs_decode_mamba2_noalloc: the Mamba-2 decode step for callers that cannot
// hand the library any device memory beyond their inputs, outputs and the
// layer state.
//
// The replay kernel needs one piece of scratch: a per-sequence arrival counter
// (rs_state.arrive) that tells the last work unit of a sequence to advance
// its pointers.  Some callers have no way to provide it: an inference-engine
// plugin whose host framework only passes the tensors it planned up front,
// or a runtime that forbids device allocation once serving starts because
// its memory plan is fixed.  This entry point keeps those counters in a
// file-scope device array instead, so it needs (and allocates) nothing.
//
// Limits and behaviour, stated for users of this entry point:
//  * at most kStaticMaxSeqs (4096) sequences per call; larger B returns
//    RS_ERR_STATIC_LIMIT before anything is enqueued;
//  * the array exists once per device that loads the library and lives until
//    the process exits (16 KiB);
//  * the first call on a device looks up the array's device address
//    (cudaGetSymbolAddress) with that device current; make that first call
//    before any stream capture;
//  * every call clears the counters it uses (cudaMemsetAsync on the caller's
//    stream) and then launches the same kernel as rs_decode_mamba2;
//  * all calls share the one array, so calls that overlap on the GPU (other
//    streams, other layers in flight at the same time) race: serialise them;
//  * no cudaMalloc, cudaFree or allocating library routine is called.
#include <mutex>

#include <cuda_runtime.h>

#include "rs.h"
#include "rs_common.cuh"
#include "rs_internal.h"

namespace {

constexpr int kStaticMaxSeqs = RS_STATIC_MAX_SEQS;
constexpr int kMaxDevices = 64;

// Zero-initialised when the module loads on a device; cleared again per call.
static __device__ __align__(256) uint32_t g_arrive[kStaticMaxSeqs];

std::mutex g_mu;
uint32_t *g_arrive_addr[kMaxDevices] = {};

// Device address of g_arrive on the current device (looked up once per device).
rs_status static_arrive(uint32_t **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return RS_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return RS_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_arrive_addr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_arrive) != cudaSuccess || !ptr) return RS_ERR_CUDA;
        g_arrive_addr[dev] = static_cast<uint32_t *>(ptr);
    }
    *out = g_arrive_addr[dev];
    return RS_OK;
}

inline bool aligned(const void *p, size_t a) { return p && (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" rs_status rs_decode_mamba2_noalloc(const rs_layer_desc *d, const rs_state *st, const uint16_t *x,
                                              const float *dt, const float *A, const uint16_t *Bm,
                                              const uint16_t *Cm, const float *D, float *y, void *stream) {
    rs_state_bytes sizes;
    const rs_status ds = rs_state_bytes_for(d, &sizes);  // validates the descriptor
    if (ds != RS_OK) return ds;
    if (d->kind != RS_MAMBA2) return RS_ERR_INVALID_ARG;
    if (d->B > kStaticMaxSeqs) return RS_ERR_STATIC_LIMIT;
    if (!st) return RS_ERR_INVALID_ARG;
    const bool need_hp = d->precision != RS_PREC_SHARED_BF16, need_lp = d->precision != RS_PREC_FP32;
    if (need_hp != (st->ckpt_hp != nullptr) || need_lp != (st->ckpt_lp != nullptr)) return RS_ERR_INVALID_ARG;
    if ((need_hp && !aligned(st->ckpt_hp, 16)) || (need_lp && !aligned(st->ckpt_lp, 16))) return RS_ERR_INVALID_ARG;
    if (!aligned(st->buf_v, 16) || !aligned(st->buf_k, 16) || !aligned(st->buf_a, 4) || !aligned(st->buf_s, 4) ||
        !aligned(st->base, 4) || !aligned(st->h, 4) || !aligned(st->nd, 4) || !aligned(st->status, 4))
        return RS_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(dt, 4) || !aligned(A, 4) || !aligned(Bm, 16) || !aligned(Cm, 16) ||
        (D && !aligned(D, 4)) || !aligned(y, 16))
        return RS_ERR_INVALID_ARG;

    uint32_t *arrive = nullptr;
    const rs_status as = static_arrive(&arrive);
    if (as != RS_OK) return as;
    cudaStream_t s = (cudaStream_t)stream;
    if (cudaMemsetAsync(arrive, 0, sizeof(uint32_t) * (size_t)d->B, s) != cudaSuccess) return RS_ERR_CUDA;

    rs::ReplayParams p = {};
    p.B = d->B; p.H = d->H; p.G = d->G; p.L = d->L; p.cap = d->capacity; p.T = 1;
    p.prec = d->precision; p.mode = rs::MODE_DECODE;
    p.ckpt_hp = st->ckpt_hp; p.ckpt_lp = st->ckpt_lp;
    p.buf_v = st->buf_v; p.buf_k = st->buf_k; p.buf_a = st->buf_a; p.buf_s = st->buf_s;
    p.base = st->base; p.h = st->h; p.nd = st->nd; p.arrive = arrive; p.status = st->status;
    p.x = x; p.dt = dt; p.A = A; p.Bm = Bm; p.Cm = Cm; p.D = D; p.y = y;
    return rs::replay_launch(p, d->kind, d->P, d->N, s) == cudaSuccess ? RS_OK : RS_ERR_CUDA;
}
