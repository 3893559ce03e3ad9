// Mamba-2 replay launches for 64 x 128 slabs (headdim 64, dstate 128), all on
// the row-split pipeline.  Verify rounds run 4 consumer warps per CTA with
// half-slab (16 KiB) stages, so that several CTAs share an SM and overlap their
// per-unit phases: three per SM up to 4 drafts, two for 5..8.  One step (and
// flush, materialise) does the same, three CTAs per SM with three stages and 4
// heads per unit, where that shape fits the buffer capacity and the batch gives
// every CTA several units; otherwise (small batches, long windows) it keeps 8
// consumer warps, whole-slab stages and two CTAs per SM.  B = 256, same GPU,
// against the 8-warp shape: one step 0.1779 against 0.1806 ms, 4 drafts 0.257
// against 0.287 ms per round, 8 drafts 0.567 against 0.615 ms; but one step at
// B = 32 0.727 against 0.744 of the copy peak and at L = 32 0.738 against 0.849.
// Rounds of 5..8 drafts also measured faster here than on the column split
// (0.485 against 0.632 ms at T = 5, 0.616 against 0.734 ms at T = 8).
#include "rs_replay_rows.cuh"

namespace rs {

namespace {
using StepCfg = rows::PipeCfg<RS_MAMBA2, 64, 128, 4, 1, 128, 3, 2>;  // 4 heads, 4 warps, 3 half-slab stages
constexpr int kStepMinBatch = 64;
}  // namespace

cudaError_t replay_launch_m2_64x128(const ReplayParams &p, cudaStream_t s) {
    const int T = p.mode == MODE_VERIFY ? p.T : 1;
    if (T > 4) return rows::launch_shape<RS_MAMBA2, 64, 128, 128, 8, 2, 8, 4, 2, 1>(p, s);
    if (T > 1) return rows::launch_shape<RS_MAMBA2, 64, 128, 128, 4, 2, 8, 4, 2, 1>(p, s);
    if (p.B >= kStepMinBatch && (p.H / p.G) % StepCfg::HU == 0 &&
        rows::pipe_smem<StepCfg>(p.cap).total <= rows::kThreePerSm)
        return rows::launch_pipe<StepCfg>(p, s);
    return rows::launch_shape<RS_MAMBA2, 64, 128, 256, 1, 1, 8, 4, 2, 1>(p, s);
}

}  // namespace rs
