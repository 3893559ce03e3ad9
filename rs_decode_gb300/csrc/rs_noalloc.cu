// rs_decode_mamba2_noalloc: the Mamba-2 decode step for callers that cannot
// hand the library any device memory beyond their inputs, outputs and the
// layer state.
//
// The replay kernel needs one piece of scratch: a per-sequence arrival counter
// (rs_state.arrive) that tells the last work unit of a sequence to advance
// its pointers, followed by the launch's two unit-scheduling counters.  Some
// callers have no way to provide it: an inference-engine plugin whose host
// framework only passes the tensors it planned up front,
// or a runtime that forbids device allocation once serving starts because
// its memory plan is fixed.  This entry point keeps those counters in a
// file-scope device array instead, so it needs (and allocates) nothing.
//
// Limits and behaviour, stated for users of this entry point:
//  * at most kStaticMaxSeqs (4096) sequences per call; larger B returns
//    RS_ERR_STATIC_LIMIT before anything is enqueued;
//  * the array exists once per device that loads the library and lives until
//    the process exits (16 KiB + 8 bytes);
//  * the first call in a device context looks up the array's device address
//    (cudaGetSymbolAddress) with that device current; make that first call
//    before any stream capture.  The address is cached per device and tagged
//    with the context's unique ID, so a call in a new context of the device
//    (after cudaDeviceReset, say) looks it up again;
//  * every call clears the counters it uses (cudaMemsetAsync on the caller's
//    stream) and then launches the same kernel as rs_decode_mamba2;
//  * all calls share the one array, so calls that overlap on the GPU (other
//    streams, other layers in flight at the same time) race: serialise them;
//  * no cudaMalloc, cudaFree or allocating library routine is called.
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "rs.h"
#include "rs_common.cuh"
#include "rs_internal.h"

namespace {

constexpr int kStaticMaxSeqs = RS_STATIC_MAX_SEQS;

// Zero-initialised when the module loads on a device; cleared again per call.
// kStaticMaxSeqs arrival counters and the two scheduling counters.
static __device__ __align__(256) uint32_t g_arrive[kStaticMaxSeqs + 2];

// The current context's unique ID (cuCtxGetCurrent + cuCtxGetId, fetched from
// the driver through the runtime: no link-time dependency on the driver
// library).  0 when it cannot be read.
using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

template <class Fn>
Fn driver_fn(const char *name) {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion(name, &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<Fn>(f);
}

unsigned long long current_context_id() {
    static const CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
    static const CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

struct ArriveAddr {
    unsigned long long ctx_id;  // context the address was looked up in
    uint32_t *addr;
};

std::mutex g_mu;
ArriveAddr g_arrive_addr[rs::kMaxDevices] = {};

// Device address of g_arrive on the current device, looked up once per device
// context.
rs_status static_arrive(uint32_t **out) {
    int dev = 0;
    rs_status st = rs::cuda_status(cudaGetDevice(&dev));
    if (st != RS_OK) return st;
    if (dev < 0 || dev >= rs::kMaxDevices) return RS_ERR_UNSUPPORTED;
    const unsigned long long ctx = current_context_id();
    std::lock_guard<std::mutex> lock(g_mu);
    ArriveAddr &a = g_arrive_addr[dev];
    if (!a.addr || ctx == 0 || a.ctx_id != ctx) {
        void *ptr = nullptr;
        st = rs::cuda_status(cudaGetSymbolAddress(&ptr, g_arrive));
        if (st != RS_OK) return st;
        if (!ptr) return RS_ERR_CUDA;
        a.addr = static_cast<uint32_t *>(ptr);
        a.ctx_id = ctx;
    }
    *out = a.addr;
    return RS_OK;
}

}  // namespace

extern "C" rs_status rs_decode_mamba2_noalloc(const rs_layer_desc *d, const rs_state *st, const uint16_t *x,
                                              const float *dt, const float *A, const uint16_t *Bm,
                                              const uint16_t *Cm, const float *D, float *y, void *stream) {
    rs_status s = rs::check_desc(d);
    if (s != RS_OK) return s;
    if (d->kind != RS_MAMBA2) return RS_ERR_INVALID_ARG;
    if (d->B > kStaticMaxSeqs) return RS_ERR_STATIC_LIMIT;
    if ((s = rs::check_state(d, st, /*need_arrive=*/false)) != RS_OK) return s;
    rs_inputs in = {};
    in.x = x; in.dt = dt; in.A = A; in.Bm = Bm; in.Cm = Cm; in.D = D;
    if ((s = rs::check_inputs(RS_MAMBA2, &in, true)) != RS_OK) return s;
    if (!y || (reinterpret_cast<uintptr_t>(y) & 15) != 0) return RS_ERR_INVALID_ARG;

    uint32_t *arrive = nullptr;
    if ((s = static_arrive(&arrive)) != RS_OK) return s;
    cudaStream_t cs = (cudaStream_t)stream;
    if ((s = rs::cuda_status(cudaMemsetAsync(arrive, 0, sizeof(uint32_t) * ((size_t)d->B + 2), cs))) != RS_OK)
        return s;

    rs::ReplayParams p = {};
    p.B = d->B; p.H = d->H; p.G = d->G; p.L = d->L; p.cap = d->capacity; p.T = 1;
    p.prec = d->precision; p.u16 = 0; p.mode = rs::MODE_DECODE;  // (Mamba-2: no flag)
    p.ckpt_hp = st->ckpt_hp; p.ckpt_lp = st->ckpt_lp;
    p.buf_v = st->buf_v; p.buf_k = st->buf_k; p.buf_a = st->buf_a; p.buf_s = st->buf_s;
    p.base = st->base; p.h = st->h; p.nd = st->nd; p.arrive = arrive; p.status = st->status;
    p.x = x; p.dt = dt; p.A = A; p.Bm = Bm; p.Cm = Cm; p.D = D; p.y = y;
    return rs::cuda_status(rs::replay_launch(p, d->kind, d->P, d->N, cs));
}
