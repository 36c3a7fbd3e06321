// k_attn.cu -- the standalone split-K decode attention kernel (device code in attn_dev.cuh).
#include "attn_dev.cuh"

namespace syn {

namespace {

template <int HD, int GP>
__global__ void __launch_bounds__(kAttnThreads) k_attn(const AttnParams p) {
    extern __shared__ __align__(16) float smem[];
    attn_prefetch(p, blockIdx.x, blockIdx.y, blockIdx.z);
    pdl_launch_dependents();
    pdl_wait();
    attn_compute<HD, GP>(p, blockIdx.x, blockIdx.y, blockIdx.z, smem);
}

template <int HD, int GP> void launch_t(const AttnParams &p, cudaStream_t s, bool pdl) {
    constexpr size_t smem = attn_smem_bytes<HD, GP>();
    if (smem > 48 * 1024) {
        static bool attr = false;
        if (!attr) {
            cudaFuncSetAttribute(k_attn<HD, GP>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            attr = true;
        }
    }
    if (pdl)
        launch_pdl(k_attn<HD, GP>, dim3(p.n_kv, p.splits, p.rows), dim3(kAttnThreads), smem, s, p);
    else
        k_attn<HD, GP><<<dim3(p.n_kv, p.splits, p.rows), kAttnThreads, smem, s>>>(p);
}

template <int HD> void launch_hd(const AttnParams &p, cudaStream_t s, bool pdl) {
    const int G = p.n_head / p.n_kv;
    if (G <= 1) return launch_t<HD, 1>(p, s, pdl);
    if (G <= 2) return launch_t<HD, 2>(p, s, pdl);
    if (G <= 4) return launch_t<HD, 4>(p, s, pdl);
    if constexpr (HD <= 128) return launch_t<HD, 8>(p, s, pdl);  // head_dim 256 allows G <= 4 (checked at create)
}

}  // namespace

void launch_attention(const AttnParams &p, cudaStream_t s) {
    switch (p.hd) {
    case 64: return launch_hd<64>(p, s, true);
    case 128: return launch_hd<128>(p, s, true);
    case 256: return launch_hd<256>(p, s, true);
    }
}

void launch_attention_ordered(const AttnParams &p, cudaStream_t s) {
    switch (p.hd) {
    case 64: return launch_hd<64>(p, s, false);
    case 128: return launch_hd<128>(p, s, false);
    case 256: return launch_hd<256>(p, s, false);
    }
}

}  // namespace syn
