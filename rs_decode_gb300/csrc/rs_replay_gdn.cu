// Gated DeltaNet replay launches for 128 x 128 slabs (d_k = d_v = 128): the
// value heads of a key head per work unit, each 64 KiB slab streamed as two
// 32 KiB row blocks through the stage ring.
#include "rs_replay.cuh"

namespace rs {

cudaError_t replay_launch_gdn_128x128(const ReplayParams &p, cudaStream_t s) {
    return dispatch_shape<RS_GDN, 128, 128, 256, 2, 2, 1>(p, s);
}

}  // namespace rs
