// Internal interface between the C-ABI entry points (rs_api.cu) and the
// kernel translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "rs.h"

namespace rs {

// Devices a process may drive through the library (ordinals 0 .. kMaxDevices-1).
constexpr int kMaxDevices = 64;

// Dynamic shared-memory opt-in of one kernel instantiation, per device.
// cudaFuncSetAttribute acts on the current device only, so each device gets
// its own grant; the mutex makes the first launches from several host threads
// safe.  This (and the per-device attribute cache of the column-split launcher)
// is the only state the library keeps between calls.
struct SmemGrants {
    std::mutex mu;
    int bytes[kMaxDevices] = {};
};

// Grants `kern` at least `smem` bytes of dynamic shared memory on the current
// device (once per device and size).
inline cudaError_t grant_smem(const void *kern, int smem, SmemGrants &g) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g.mu);
    if (g.bytes[dev] < smem) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        g.bytes[dev] = smem;
    }
    return cudaSuccess;
}

// Host-side checks shared by the entry points (rs_api.cu).  check_state with
// need_arrive = false ignores the arrival-counter array (the entry point that
// keeps its own counters).
rs_status check_desc(const rs_layer_desc *d);
rs_status check_state(const rs_layer_desc *d, const rs_state *s, bool need_arrive = true);
rs_status check_inputs(int kind, const rs_inputs *in, bool need_q);
// RS_OK for cudaSuccess; otherwise records the error's name and text for
// rs_last_cuda_error (per host thread) and returns RS_ERR_CUDA.
rs_status cuda_status(cudaError_t e);

// Arguments of the replay kernels (decode, verify, flush, materialise).
struct ReplayParams {
    int B, H, G, L, cap, T, prec, mode;
    int u16;     // GDN records keep u in bf16 (RS_U_BF16)
    float *ckpt_hp;
    uint16_t *ckpt_lp;
    void *buf_v;
    uint16_t *buf_k;
    float *buf_a, *buf_s;
    int32_t *base, *h, *nd;
    uint32_t *arrive, *status;
    // step / draft inputs, [B][T][...]
    const uint16_t *x;
    const float *dt, *A;
    const uint16_t *Bm, *Cm;
    const float *D;
    const uint16_t *q, *k, *v;
    const float *alpha, *beta;
    float *y;    // outputs [B][T][H][P]
    float *out;  // materialise destination [B][H][N][P]
};

// Arguments of the eager (load-update-store) baselines.
struct EagerParams {
    int B, H, G, T, slots;  // slots: pool slots per sequence (verify), 1 for a plain step
    float *S;               // state (plain step) or snapshot pool (verify)
    const int32_t *cur;     // pool slot of the committed state (verify), may be null
    const uint16_t *x;
    const float *dt, *A;
    const uint16_t *Bm, *Cm;
    const float *D;
    const uint16_t *q, *k, *v;
    const float *alpha, *beta;
    float *y;
};

bool replay_shape_supported(int kind, int P, int N);
cudaError_t replay_launch(const ReplayParams &p, int kind, int P, int N, cudaStream_t s);
// Per family / slab shape (one translation unit each, compiled in parallel).
cudaError_t replay_launch_m2_64x128(const ReplayParams &p, cudaStream_t s);
cudaError_t replay_launch_gdn_128x128(const ReplayParams &p, cudaStream_t s);
cudaError_t replay_launch_kda_128x128(const ReplayParams &p, cudaStream_t s);
cudaError_t replay_launch_64x64(const ReplayParams &p, int kind, cudaStream_t s);
// Small-batch Mamba-2 decode with the fp32 checkpoint: one CTA per two heads,
// no pipeline (rs_replay_direct.cu).
bool replay_direct_applies(const ReplayParams &p, int kind, int P, int N);
cudaError_t replay_direct_launch(const ReplayParams &p, cudaStream_t s);
cudaError_t eager_launch(const EagerParams &p, int kind, int P, int N, cudaStream_t s);

// Small kernels (rs_small.cu).
cudaError_t init_launch(const rs_layer_desc &d, const rs_state &st, const float *init, cudaStream_t s);
cudaError_t commit_launch(int B, const int32_t *accepted, int32_t *h, int32_t *nd, uint32_t *status,
                          cudaStream_t s);
cudaError_t rollback_launch(int B, int32_t *nd, cudaStream_t s);
cudaError_t append_launch(const rs_layer_desc &d, const rs_state &st, int n, const rs_inputs &in,
                          cudaStream_t s);
cudaError_t select_launch(int B, int slots, int32_t *cur, const int32_t *accepted, uint32_t *status,
                          cudaStream_t s);

}  // namespace rs
