// k_misc.cu -- standalone kernels for the small ops (device code in misc_dev.cuh): embed,
// rms_norm, the elementwise ops, the per-head transforms with the KV append, and the greedy argmax
// of the logits ("Local inference and architectures", section "The operations").
#include <algorithm>
#include <map>
#include <mutex>
#include <tuple>

#include "misc_dev.cuh"

namespace syn {

namespace {

__global__ void k_embed(const EmbedParams p) {
    pdl_launch_dependents();
    pdl_wait();
    embed_cta(p, blockIdx.x, gridDim.x);
}

__global__ void k_rmsnorm(const RmsParams p) {
    __shared__ float red[32];
    pdl_launch_dependents();
    pdl_wait();
    rms_cta(p, blockIdx.x, gridDim.x, red);
}

__global__ void k_eltwise(const EltParams p) {
    pdl_launch_dependents();
    pdl_wait();
    elt_cta(p, blockIdx.x, gridDim.x);
}

// Unlike the other kernels, this one lets its dependents start only after its own wait: the
// attention kernel that follows it streams the old cache positions before it waits, using the
// step's position from the device state, and relies on every kernel before this one (the previous
// step's argmax included) having completed when it starts.
__global__ void k_heads(const HeadsParams p) {
    pdl_wait();
    pdl_launch_dependents();
    heads_cta(p, blockIdx.x, gridDim.x);
}

__global__ void k_argmax(const ArgmaxParams p) {
    __shared__ float sv[32];
    __shared__ int si[32];
    __shared__ int last;
    pdl_launch_dependents();
    pdl_wait();
    argmax_cta(p, blockIdx.x, gridDim.x, sv, si, &last);
}

__global__ void k_dequant_rows(const DevMatrix W, int row0, int nrows, float *out) {
    pdl_launch_dependents();
    pdl_wait();
    const int64_t n = (int64_t)nrows * W.K;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        out[i] = dequant_one(W, row0 + i / W.K, i % W.K);
}


}  // namespace

cudaError_t ensure_dyn_smem(const void *func, int bytes) {
    static std::mutex mu;
    static std::map<std::pair<const void *, int>, int> done;   // (kernel, device) -> size set
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    auto it = done.find({func, dev});
    if (it != done.end() && it->second >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done[{func, dev}] = bytes;
    return e;
}

void launch_embed(const EmbedParams &p, cudaStream_t s) {
    const int64_t n = (int64_t)p.n * p.E.K;
    launch_pdl(k_embed, dim3((unsigned)std::min<int64_t>((n + 255) / 256, 4096)), dim3(256), 0, s, p);
}

void launch_rmsnorm(const RmsParams &p, cudaStream_t s) { launch_pdl(k_rmsnorm, dim3(p.rows), dim3(256), 0, s, p); }

void launch_eltwise(const EltParams &p, cudaStream_t s) {
    const int64_t n = (int64_t)p.rows * p.width;
    const int blocks = (int)std::min<int64_t>((n + 1023) / 1024, 152 * 8);
    launch_pdl(k_eltwise, dim3(blocks), dim3(256), 0, s, p);
}

void launch_heads(const HeadsParams &p, cudaStream_t s) {
    const int warps = (p.nq + p.nk) * p.rows;
    const int blocks = (warps * 32 + 127) / 128;
    launch_pdl(k_heads, dim3(blocks), dim3(128), 0, s, p);
}

void launch_argmax(const ArgmaxParams &p, int blocks, cudaStream_t s) { launch_pdl(k_argmax, dim3(blocks), dim3(512), 0, s, p); }

void launch_copy_row(float *dst, const float *src, int width, cudaStream_t s) {
    cudaMemcpyAsync(dst, src, (size_t)width * sizeof(float), cudaMemcpyDeviceToDevice, s);
}

void launch_dequant_rows(const DevMatrix &W, int row0, int nrows, float *out, cudaStream_t s) {
    const int64_t n = (int64_t)nrows * W.K;
    const int blocks = (int)std::min<int64_t>((n + 255) / 256, 8192);
    launch_pdl(k_dequant_rows, dim3(blocks), dim3(256), 0, s, W, row0, nrows, out);
}

}  // namespace syn
