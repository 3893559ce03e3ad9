// Gated DeltaNet replay launches for 128 x 128 slabs (d_k = d_v = 128): the
// column-split pipeline, four 16 KiB row blocks per fp32 slab, two per bf16
// slab.
#include "rs_replay_cols.cuh"

namespace rs {

cudaError_t replay_launch_gdn_128x128(const ReplayParams &p, cudaStream_t s) {
    return cols::dispatch_shape<RS_GDN, 128, 128>(p, s);
}

}  // namespace rs
