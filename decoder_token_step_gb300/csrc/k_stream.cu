// k_stream.cu -- shared-memory sizes and the cooperative launch of the persistent streaming
// decode-step kernel (device code in k_stream.cuh, one instantiation per k_stream_<head dim>_<group>.cu).
#include "attn_dev.cuh"
#include "gemv_dev.cuh"
#include "syn_internal.h"
#include "misc_dev.cuh"

namespace syn {

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

// the instantiations live in k_stream_<head dim>_<group>.cu (compiled in parallel)
const void *stream_kernel_64_1();
const void *stream_kernel_64_2();
const void *stream_kernel_64_4();
const void *stream_kernel_64_8();
const void *stream_kernel_128_1();
const void *stream_kernel_128_2();
const void *stream_kernel_128_4();
const void *stream_kernel_128_8();
const void *stream_kernel_256_1();
const void *stream_kernel_256_2();
const void *stream_kernel_256_4();

namespace {

const void *stream_kernel(int hd, int gp) {
    switch (hd * 16 + gp) {
    case 64 * 16 + 1: return stream_kernel_64_1();
    case 64 * 16 + 2: return stream_kernel_64_2();
    case 64 * 16 + 4: return stream_kernel_64_4();
    case 64 * 16 + 8: return stream_kernel_64_8();
    case 128 * 16 + 1: return stream_kernel_128_1();
    case 128 * 16 + 2: return stream_kernel_128_2();
    case 128 * 16 + 4: return stream_kernel_128_4();
    case 128 * 16 + 8: return stream_kernel_128_8();
    case 256 * 16 + 1: return stream_kernel_256_1();
    case 256 * 16 + 2: return stream_kernel_256_2();
    case 256 * 16 + 4: return stream_kernel_256_4();
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
    cfg.blockDim = dim3(kStreamBlockThreads);   // the consumer warps, the producer and the publisher warp
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
