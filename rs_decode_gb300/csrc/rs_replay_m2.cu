// Mamba-2 replay launches for 64 x 128 slabs (headdim 64, dstate 128): the
// row-split pipeline, 8, 4, 2 or 1 heads per work unit, 32 KiB stages.
#include "rs_replay_rows.cuh"

namespace rs {

cudaError_t replay_launch_m2_64x128(const ReplayParams &p, cudaStream_t s) {
    return rows::dispatch_shape<RS_MAMBA2, 64, 128, 256, 1, 8, 4, 2, 1>(p, s);
}

}  // namespace rs
