// Mamba-2 replay launches for 64 x 128 slabs (headdim 64, dstate 128), all on
// the row-split pipeline (8, 4, 2 or 1 heads per work unit, 32 KiB stages):
// one step, and verify rounds in the draft buckets of up to 4 and of 5..8
// drafts.  (Rounds of 5..8 drafts measured faster here than on the column
// split: 0.485 against 0.632 ms at T = 5, 0.616 against 0.734 ms at T = 8,
// B = 256.)
#include "rs_replay_rows.cuh"

namespace rs {

cudaError_t replay_launch_m2_64x128(const ReplayParams &p, cudaStream_t s) {
    const int T = p.mode == MODE_VERIFY ? p.T : 1;
    if (T > 4) return rows::launch_shape<RS_MAMBA2, 64, 128, 256, 8, 1, 8, 4, 2, 1>(p, s);
    if (T > 1) return rows::launch_shape<RS_MAMBA2, 64, 128, 256, 4, 1, 8, 4, 2, 1>(p, s);
    return rows::launch_shape<RS_MAMBA2, 64, 128, 256, 1, 1, 8, 4, 2, 1>(p, s);
}

}  // namespace rs
