// k_stream.cu -- shared-memory sizes and the cooperative launch of the persistent streaming
// decode-step kernel (device code in k_stream.cuh, instantiations in k_stream_hd*.cu).
#include "attn_dev.cuh"
#include "gemv_dev.cuh"
#include "syn_internal.h"
#include "misc_dev.cuh"

namespace syn {

size_t stream_gemv_aux_bytes(int wtype, size_t row_bytes) { return gemv_smem_bytes_rt(wtype, row_bytes); }

size_t stream_attn_aux_bytes(int hd, int gp) {
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

// the instantiations live in k_stream_hd{64,128,256}.cu (compiled in parallel)
const void *stream_kernel_hd64(int gp);
const void *stream_kernel_hd128(int gp);
const void *stream_kernel_hd256(int gp);

namespace {

const void *stream_kernel(int hd, int gp) {
    switch (hd) {
    case 64: return stream_kernel_hd64(gp);
    case 128: return stream_kernel_hd128(gp);
    case 256: return stream_kernel_hd256(gp);
    }
    return nullptr;
}

}  // namespace

bool stream_supported(int hd, int gp) { return stream_kernel(hd, gp) != nullptr; }

// dynamic shared memory one CTA may take next to the kernel's static shared memory
int stream_max_dyn_smem() {
    int dev = 0, optin = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    cudaFuncAttributes fa;
    const void *fn = stream_kernel(128, 4);
    if (!fn || cudaFuncGetAttributes(&fa, fn) != cudaSuccess) return 0;
    return optin - (int)fa.sharedSizeBytes;
}

cudaError_t launch_stream(int hd, int gp, const StreamParams &sp, int blocks, cudaStream_t s) {
    const void *fn = stream_kernel(hd, gp);
    if (!fn) return cudaErrorInvalidValue;
    const int smem = sp.nslots * kSlotBytes + sp.aux_bytes + 128;   // + alignment slack of the ring
    cudaError_t e = ensure_dyn_smem(fn, smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks);
    cfg.blockDim = dim3(kConsumerThreads + 32);   // the consumer warps and the producer warp
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeCooperative;
    at[0].val.cooperative = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    void *args[] = {const_cast<StreamParams *>(&sp)};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace syn
