// k_step_q8_0.cu -- the persistent step kernel instantiated for q8_0 weights (k_step.cuh).
#include "k_step.cuh"

namespace syn {
int step_blocks_per_sm_q8_0(int hd, int gp, size_t smem) { return step_blocks_per_sm_wt<W_Q8_0>(hd, gp, smem); }
cudaError_t launch_step_q8_0(int hd, int gp, const StepParams &sp, int blocks, size_t smem, cudaStream_t s) {
    return launch_step_wt<W_Q8_0>(hd, gp, sp, blocks, smem, s);
}
}  // namespace syn
