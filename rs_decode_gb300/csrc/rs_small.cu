// Small kernels around the replay path: checkpoint initialisation (both
// precisions), commit / rollback pointer moves, append-only records, and the
// snapshot selection of the eager speculative baseline.
#include "rs_common.cuh"
#include "rs_internal.h"

namespace rs {

// ---------------------------------------------------------------- init
// Writes the fp32 and/or bf16 checkpoint from init (or zeros) and clears the
// per-sequence pointers, the arrival and scheduling counters (B + 2) and the
// status word.
__global__ void init_kernel(size_t n4, const float4 *init, float4 *hp, uint2 *lp, int B, int32_t *base,
                            int32_t *h, int32_t *nd, uint32_t *arrive, uint32_t *status) {
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride) {
        const float4 v = init ? init[i] : make_float4(0.f, 0.f, 0.f, 0.f);
        if (hp) hp[i] = v;
        if (lp) lp[i] = make_uint2(pack_bf2(v.x, v.y), pack_bf2(v.z, v.w));
    }
    for (size_t b = (size_t)blockIdx.x * blockDim.x + threadIdx.x; b < (size_t)B; b += stride) {
        base[b] = 0;
        h[b] = 0;
        nd[b] = 0;
        arrive[b] = 0;
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        arrive[B] = arrive[B + 1] = 0;
        *status = 0;
    }
}

cudaError_t init_launch(const rs_layer_desc &d, const rs_state &st, const float *init, cudaStream_t s) {
    const size_t n4 = (size_t)d.B * d.H * d.N * d.P / 4;
    const int threads = 256;
    int blocks = (int)((n4 + threads - 1) / threads);
    if (blocks > 152 * 16) blocks = 152 * 16;
    if (blocks < 1) blocks = 1;
    init_kernel<<<blocks, threads, 0, s>>>(n4, reinterpret_cast<const float4 *>(init),
                                           reinterpret_cast<float4 *>(st.ckpt_hp),
                                           reinterpret_cast<uint2 *>(st.ckpt_lp), d.B, st.base, st.h, st.nd,
                                           st.arrive, st.status);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- commit / rollback
// Accepting a prefix of the drafts only moves a pointer by the accepted count
// (the commit box of the flowchart in "ReplaySSM: Cache SSM Inputs, Not
// State"); rejected records stay in the buffer and are overwritten later.
__global__ void commit_kernel(int B, const int32_t *accepted, int32_t *h, int32_t *nd, uint32_t *status) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    const int n = nd[b];
    int a = accepted ? accepted[b] : 0;
    if (a < 0 || a > n) {
        atomicOr(status, RS_DEV_ACCEPT);
        a = a < 0 ? 0 : n;
    }
    h[b] += a;
    nd[b] = 0;
}

cudaError_t commit_launch(int B, const int32_t *accepted, int32_t *h, int32_t *nd, uint32_t *status,
                          cudaStream_t s) {
    commit_kernel<<<(B + 255) / 256, 256, 0, s>>>(B, accepted, h, nd, status);
    return cudaGetLastError();
}

__global__ void rollback_kernel(int B, int32_t *nd) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b < B) nd[b] = 0;
}

cudaError_t rollback_launch(int B, int32_t *nd, cudaStream_t s) {
    rollback_kernel<<<(B + 255) / 256, 256, 0, s>>>(B, nd);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- append (Mamba-2)
// Copies n records per sequence into slots (base + h + i) % cap; a second
// launch then advances h.  A sequence with drafts pending or without room is
// left unchanged and flagged.
__device__ __forceinline__ bool append_ok(int hc, int ndr, int n, int cap) { return ndr == 0 && hc + n <= cap; }

__global__ void append_copy_kernel(int H, int G, int P, int N, int cap, int n, const uint16_t *x,
                                   const float *dt, const float *A, const uint16_t *Bm, uint16_t *buf_x,
                                   float *buf_a, float *buf_dt, uint16_t *buf_k, const int32_t *base,
                                   const int32_t *h, const int32_t *nd) {
    const int i = blockIdx.x, b = blockIdx.y;
    const int hc = h[b];
    if (!append_ok(hc, nd[b], n, cap)) return;
    const int slot = (base[b] + hc + i) % cap;
    const size_t src_rec = (size_t)b * n + i, dst_rec = (size_t)b * cap + slot;
    const uint4 *sx = reinterpret_cast<const uint4 *>(x + src_rec * H * P);
    uint4 *dx = reinterpret_cast<uint4 *>(buf_x + dst_rec * H * P);
    for (int c = threadIdx.x; c < H * P / 8; c += blockDim.x) dx[c] = sx[c];
    const uint4 *sk = reinterpret_cast<const uint4 *>(Bm + src_rec * G * N);
    uint4 *dk = reinterpret_cast<uint4 *>(buf_k + dst_rec * G * N);
    for (int c = threadIdx.x; c < G * N / 8; c += blockDim.x) dk[c] = sk[c];
    for (int c = threadIdx.x; c < H; c += blockDim.x) {
        const float d = dt[src_rec * H + c];
        buf_dt[dst_rec * H + c] = d;
        buf_a[dst_rec * H + c] = expf(d * A[c]);
    }
}

__global__ void append_ptr_kernel(int B, int cap, int n, int32_t *h, const int32_t *nd, uint32_t *status) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    const int hc = h[b], ndr = nd[b];
    if (append_ok(hc, ndr, n, cap)) {
        h[b] = hc + n;
    } else {
        atomicOr(status, ndr ? RS_DEV_DRAFTS_PENDING : RS_DEV_CAPACITY);
    }
}

cudaError_t append_launch(const rs_layer_desc &d, const rs_state &st, int n, const rs_inputs &in,
                          cudaStream_t s) {
    append_copy_kernel<<<dim3(n, d.B), 256, 0, s>>>(d.H, d.G, d.P, d.N, d.capacity, n, in.x, in.dt, in.A, in.Bm,
                                                    static_cast<uint16_t *>(st.buf_v), st.buf_a, st.buf_s,
                                                    st.buf_k, st.base, st.h, st.nd);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    append_ptr_kernel<<<(d.B + 255) / 256, 256, 0, s>>>(d.B, d.capacity, n, st.h, st.nd, st.status);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- eager snapshot selection
__global__ void select_kernel(int B, int slots, int32_t *cur, const int32_t *accepted, uint32_t *status) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    int a = accepted[b];
    if (a < 0 || a >= slots) {
        if (status) atomicOr(status, RS_DEV_ACCEPT);
        a = a < 0 ? 0 : slots - 1;
    }
    cur[b] = (cur[b] + a) % slots;
}

cudaError_t select_launch(int B, int slots, int32_t *cur, const int32_t *accepted, uint32_t *status,
                          cudaStream_t s) {
    select_kernel<<<(B + 255) / 256, 256, 0, s>>>(B, slots, cur, accepted, status);
    return cudaGetLastError();
}

}  // namespace rs
