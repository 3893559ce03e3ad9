// Replay launches of layers with one decay per key channel (RS_KDA) for
// 128 x 128 slabs: the column-split pipeline, four 16 KiB row blocks per fp32
// slab.
#include "rs_replay_cols.cuh"

namespace rs {

cudaError_t replay_launch_kda_128x128(const ReplayParams &p, cudaStream_t s) {
    return cols::dispatch_shape<RS_KDA, 128, 128>(p, s);
}

}  // namespace rs
