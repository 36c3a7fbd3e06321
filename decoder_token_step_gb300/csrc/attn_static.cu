// attn_static.cu -- decode attention that performs no device allocation (the attention operation
// of "Local inference and architectures", section "The operations"; an entry point of this library
// with no counterpart on the pages).
//
// Some callers cannot allocate device memory at the moment they need attention: code that runs
// while a stream is being captured into a CUDA graph (allocation calls are not allowed during a
// capture), or a plug-in inside a host framework that has already reserved the device's memory for
// its own pool, so a further cudaMalloc would fail or break the host's accounting. For them,
// syn_attention_static runs the split-K decode attention kernel with its scratch (the per-split
// partial results, the completion counters and the position record) in one file-scope device array
// of fixed size that is part of the loaded library. The caller passes the query, the KV cache and the
// output buffer, all already on the device.
#include <atomic>
#include <mutex>

#include "../../include/syn.h"
#include "device_common.cuh"

using namespace syn;

namespace {

// Scratch layout: [DevState | pad to 256 B][counters: kMaxKvHeads x u32][split partials: floats].
constexpr size_t kScratchBytes = (size_t)4 << 20;  // 4 MiB on every GPU that loads the library
constexpr int kMaxKvHeads = 1024;
constexpr size_t kCountersOff = 256;
constexpr size_t kPartOff = kCountersOff + (size_t)kMaxKvHeads * sizeof(unsigned);
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_attn_scratch[kScratchBytes];

std::mutex g_mu;
void *g_scratch_addr[kMaxDevices] = {};
std::atomic<int> g_spin{-1};   // test support: polls before a wait gives up (-1 = the kernels' default bound)

// Writes the query position and clears the completion counters (they must start at zero; the
// array keeps whatever the previous call left in it). The error word is left alone: it is sticky
// until syn_attention_static_status reads and clears it.
__global__ void k_static_prepare(int pos, int n_kv) {
    unsigned *ctr = reinterpret_cast<unsigned *>(g_attn_scratch + kCountersOff);
    for (int i = threadIdx.x; i < n_kv; i += blockDim.x) ctr[i] = 0u;
    if (threadIdx.x == 0) {
        DevState *st = reinterpret_cast<DevState *>(g_attn_scratch);
        st->pos = pos;
        st->n = 1;
        st->argmax = 0;
    }
}

// This device's address of the array, looked up on the first call with the device current.
syn_status scratch_base(void **base) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SYN_E_BACKEND_INIT;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_attn_scratch) != cudaSuccess || !ptr) return SYN_E_CUDA;
        g_scratch_addr[dev] = ptr;
    }
    *base = g_scratch_addr[dev];
    return SYN_OK;
}

}  // namespace

extern "C" syn_status syn_attention_static(const float *q, const float *k_cache, const float *v_cache,
                                           int n_head, int n_head_kv, int head_dim, int max_ctx, int n_ctx,
                                           int window, int splits, float *out, void *cuda_stream) {
    if (!q || !k_cache || !v_cache || !out) return SYN_E_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128 && head_dim != 256) return SYN_E_UNSUPPORTED_OP;
    if (n_head_kv < 1 || n_head_kv > kMaxKvHeads || n_head < n_head_kv || n_head % n_head_kv) return SYN_E_INVALID_ARG;
    if (n_head / n_head_kv > (head_dim == 256 ? 4 : 8)) return SYN_E_UNSUPPORTED_OP;
    if (n_ctx < 1 || n_ctx > max_ctx || window < 0 || splits < 1 || splits > 64) return SYN_E_INVALID_ARG;
    // the cache rows are streamed with bulk copies, which need 16-byte aligned addresses
    if ((reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache)) & 15) return SYN_E_INVALID_ARG;
    const size_t part_bytes = (size_t)splits * n_head * (head_dim + 4) * sizeof(float);
    if (part_bytes > kScratchBytes - kPartOff) return SYN_E_INVALID_ARG;

    void *base = nullptr;
    const syn_status st = scratch_base(&base);
    if (st != SYN_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    k_static_prepare<<<1, 256, 0, s>>>(n_ctx - 1, n_head_kv);

    AttnParams p;
    p.q = q;
    p.ldq = (int64_t)n_head * head_dim;
    p.out = out;
    p.ldo = (int64_t)n_head * head_dim;
    p.kcache = k_cache;
    p.vcache = v_cache;
    p.n_head = n_head;
    p.n_kv = n_head_kv;
    p.hd = head_dim;
    p.max_ctx = max_ctx;
    p.rows = 1;
    p.window = window;
    p.splits = splits;
    p.state = reinterpret_cast<const DevState *>(base);
    p.err = &reinterpret_cast<DevState *>(base)->err;
    p.counters = reinterpret_cast<unsigned *>(static_cast<unsigned char *>(base) + kCountersOff);
    p.part = reinterpret_cast<float *>(static_cast<unsigned char *>(base) + kPartOff);
    p.spin = g_spin.load();
    launch_attention_ordered(p, s);
    return cudaGetLastError() == cudaSuccess ? SYN_OK : SYN_E_CUDA;
}

extern "C" syn_status syn_attention_static_status(void *cuda_stream) {
    void *base = nullptr;
    const syn_status st = scratch_base(&base);
    if (st != SYN_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
    int *err = &static_cast<DevState *>(base)->err;
    int h = 0;
    if (cudaMemcpyAsync(&h, err, sizeof h, cudaMemcpyDeviceToHost, s) != cudaSuccess) return SYN_E_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return SYN_E_CUDA;
    if (h == 0) return SYN_OK;
    if (cudaMemsetAsync(err, 0, sizeof(int), s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess) return SYN_E_CUDA;
    return SYN_E_CUDA;
}

extern "C" void syn_debug_set_spin_limit(int polls) { g_spin.store(polls < 0 ? -1 : polls); }
