// k_step.cu -- dispatch of the persistent step kernel by weight type, and host-side size helpers.
#include "attn_dev.cuh"
#include "gemv_dev.cuh"

namespace syn {

int step_blocks_per_sm_f32(int hd, int gp, size_t smem);
int step_blocks_per_sm_f16(int hd, int gp, size_t smem);
int step_blocks_per_sm_q8_0(int hd, int gp, size_t smem);
int step_blocks_per_sm_q4_0(int hd, int gp, size_t smem);
cudaError_t launch_step_f32(int hd, int gp, const StepParams &sp, int blocks, size_t smem, cudaStream_t s);
cudaError_t launch_step_f16(int hd, int gp, const StepParams &sp, int blocks, size_t smem, cudaStream_t s);
cudaError_t launch_step_q8_0(int hd, int gp, const StepParams &sp, int blocks, size_t smem, cudaStream_t s);
cudaError_t launch_step_q4_0(int hd, int gp, const StepParams &sp, int blocks, size_t smem, cudaStream_t s);

int step_blocks_per_sm(int wtype, int hd, int gp, size_t smem) {
    switch (wtype) {
    case W_F32: return step_blocks_per_sm_f32(hd, gp, smem);
    case W_F16: return step_blocks_per_sm_f16(hd, gp, smem);
    case W_Q8_0: return step_blocks_per_sm_q8_0(hd, gp, smem);
    case W_Q4_0: return step_blocks_per_sm_q4_0(hd, gp, smem);
    }
    return 0;
}

cudaError_t launch_step(int wtype, int hd, int gp, const StepParams &sp, int blocks, size_t smem, cudaStream_t s) {
    switch (wtype) {
    case W_F32: return launch_step_f32(hd, gp, sp, blocks, smem, s);
    case W_F16: return launch_step_f16(hd, gp, sp, blocks, smem, s);
    case W_Q8_0: return launch_step_q8_0(hd, gp, sp, blocks, smem, s);
    case W_Q4_0: return launch_step_q4_0(hd, gp, sp, blocks, smem, s);
    }
    return cudaErrorInvalidValue;
}

size_t gemv_smem_bytes_host(int wtype, size_t row_bytes) { return gemv_smem_bytes_rt(wtype, row_bytes); }

size_t attn_smem_bytes_host(int hd, int gp) {
    switch (hd * 16 + gp) {
    case 64 * 16 + 1: return attn_smem_bytes<64, 1>();
    case 64 * 16 + 2: return attn_smem_bytes<64, 2>();
    case 64 * 16 + 4: return attn_smem_bytes<64, 4>();
    case 64 * 16 + 8: return attn_smem_bytes<64, 8>();
    case 128 * 16 + 1: return attn_smem_bytes<128, 1>();
    case 128 * 16 + 2: return attn_smem_bytes<128, 2>();
    case 128 * 16 + 4: return attn_smem_bytes<128, 4>();
    case 128 * 16 + 8: return attn_smem_bytes<128, 8>();
    case 256 * 16 + 1: return attn_smem_bytes<256, 1>();
    case 256 * 16 + 2: return attn_smem_bytes<256, 2>();
    case 256 * 16 + 4: return attn_smem_bytes<256, 4>();
    }
    return 0;
}

}  // namespace syn
