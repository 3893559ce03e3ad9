// Mamba-2 replay launches for 64 x 128 slabs (headdim 64, dstate 128).  One
// step and verify rounds of up to 4 drafts run on the row-split pipeline
// (8, 4, 2 or 1 heads per work unit, 32 KiB stages); rounds of 5..8 drafts,
// whose 8 dot vectors per element need the registers of warp-local column
// ownership, run on the column-split pipeline.
#include "rs_replay_cols.cuh"
#include "rs_replay_rows.cuh"

namespace rs {

cudaError_t replay_launch_m2_64x128(const ReplayParams &p, cudaStream_t s) {
    const int T = p.mode == MODE_VERIFY ? p.T : 1;
    if (T > 4) return cols::launch_pipe<cols::RCfg<RS_MAMBA2, 64, 128, 8>>(p, s);
    if (T > 1) return rows::launch_shape<RS_MAMBA2, 64, 128, 256, 4, 1, 8, 4, 2, 1>(p, s);
    return rows::launch_shape<RS_MAMBA2, 64, 128, 256, 1, 1, 8, 4, 2, 1>(p, s);
}

}  // namespace rs
