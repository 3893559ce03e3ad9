// Internal interface between the C-ABI entry points (rs_api.cu) and the
// kernel translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "rs.h"

namespace rs {

// Arguments of the replay kernels (decode, verify, flush, materialise).
struct ReplayParams {
    int B, H, G, L, cap, T, prec, mode;
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
cudaError_t replay_launch_64x64(const ReplayParams &p, int kind, cudaStream_t s);
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
