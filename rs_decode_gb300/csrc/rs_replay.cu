// Replay launch entry: dispatch on the layer family and slab shape, plus the
// small 64 x 64 slab shapes of both families.
#include "rs_replay.cuh"

namespace rs {

cudaError_t replay_launch_64x64(const ReplayParams &p, int kind, cudaStream_t s) {
    if (kind == RS_MAMBA2) return dispatch_shape<RS_MAMBA2, 64, 64, 128, 1, 2, 1>(p, s);
    return dispatch_shape<RS_GDN, 64, 64, 128, 1, 2, 1>(p, s);
}

cudaError_t replay_launch(const ReplayParams &p, int kind, int P, int N, cudaStream_t s) {
    if (kind == RS_MAMBA2 && P == 64 && N == 128) return replay_launch_m2_64x128(p, s);
    if (kind == RS_GDN && P == 128 && N == 128) return replay_launch_gdn_128x128(p, s);
    if (P == 64 && N == 64) return replay_launch_64x64(p, kind, s);
    return cudaErrorInvalidValue;
}

bool replay_shape_supported(int kind, int P, int N) {
    if (kind == RS_MAMBA2) return P == 64 && (N == 128 || N == 64);
    return (P == 128 && N == 128) || (P == 64 && N == 64);
}

}  // namespace rs
