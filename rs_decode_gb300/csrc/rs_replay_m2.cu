// Mamba-2 replay launches for 64 x 128 slabs (headdim 64, dstate 128), all on
// the row-split pipeline.  One step: 8 consumer warps, whole-slab (32 KiB)
// stages, two CTAs per SM.  Verify rounds (the draft buckets of up to 4 and of
// 5..8 drafts): 4 consumer warps and half-slab (16 KiB) stages, so that three
// CTAs (two for 8 drafts) share an SM and overlap their per-unit phases
// (B = 256, same box: 4 drafts 0.257 against 0.287 ms per round, 8 drafts
// 0.567 against 0.615 ms; one step 0.1818 against 0.1801 ms, so it keeps the
// wider CTAs).  Rounds of 5..8 drafts measured faster here than on the column
// split (0.485 against 0.632 ms at T = 5, 0.616 against 0.734 ms at T = 8).
#include "rs_replay_rows.cuh"

namespace rs {

cudaError_t replay_launch_m2_64x128(const ReplayParams &p, cudaStream_t s) {
    const int T = p.mode == MODE_VERIFY ? p.T : 1;
    if (T > 4) return rows::launch_shape<RS_MAMBA2, 64, 128, 128, 8, 2, 8, 4, 2, 1>(p, s);
    if (T > 1) return rows::launch_shape<RS_MAMBA2, 64, 128, 128, 4, 2, 8, 4, 2, 1>(p, s);
    return rows::launch_shape<RS_MAMBA2, 64, 128, 256, 1, 1, 8, 4, 2, 1>(p, s);
}

}  // namespace rs
