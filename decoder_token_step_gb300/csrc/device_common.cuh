// device_common.cuh -- small device helpers of the libsyn kernels (weight decoding, reductions,
// streaming loads). Internal to the CUDA sources.
#pragma once

#include <cuda_fp16.h>
#include <cstdint>
#include <utility>

#include "syn_internal.h"

namespace syn {

#define SYN_DEV __device__ __forceinline__

// 128-bit load of data read exactly once (weights): no L1 allocation.
SYN_DEV uint4 ld_stream16(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

SYN_DEV uint16_t ld_stream2(const void *p) {
    unsigned short r;
    asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(r) : "l"(p));
    return r;
}

SYN_DEV float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

SYN_DEV float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

SYN_DEV float half_bits_to_float(uint16_t h) { return __half2float(__ushort_as_half(h)); }

// Programmatic dependent launch: a kernel launched with launch_pdl may start while the previous
// kernel on the stream is still running. Everything before pdl_wait() must touch only data that no
// earlier kernel of the step writes (weights, old KV positions); pdl_wait() returns once the
// previous kernel has completed and its writes are visible. Without the launch attribute both are
// no-ops.
SYN_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
SYN_DEV void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }

template <typename... KArgs, typename... Args>
inline void launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Dequantised value of element k of row `row` of W (f32; exact: d * code).
SYN_DEV float dequant_one(const DevMatrix &W, int64_t row, int64_t k) {
    const uint8_t *rp = reinterpret_cast<const uint8_t *>(W.codes) + (size_t)row * W.row_bytes;
    switch (W.wtype) {
    case W_F32: return reinterpret_cast<const float *>(rp)[k];
    case W_F16: return half_bits_to_float(reinterpret_cast<const uint16_t *>(rp)[k]);
    case W_Q8_0: {
        // codes are stored offset-binary (q + 128)
        float d = half_bits_to_float(W.scales[(size_t)row * W.scale_stride + k / 32]);
        return d * (float)((int)rp[k] - 128);
    }
    case W_Q4_0: {
        float d = half_bits_to_float(W.scales[(size_t)row * W.scale_stride + k / 32]);
        int64_t blk = k / 32, j = k % 32;
        uint8_t byte = rp[blk * 16 + (j & 15)];
        int code = j < 16 ? (byte & 15) : (byte >> 4);
        return d * (float)(code - 8);
    }
    }
    return 0.f;
}

SYN_DEV float apply_act(int act, float g) {
    switch (act) {
    case ACT_SILU: return g / (1.f + expf(-g));
    case ACT_GELU: return 0.5f * g * (1.f + erff(g * 0.70710678118654752f));
    case ACT_GELU_TANH: {
        const float c = 0.79788456080286536f;  // sqrt(2/pi)
        return 0.5f * g * (1.f + tanhf(c * (g + 0.044715f * g * g * g)));
    }
    case ACT_RELU: return g > 0.f ? g : 0.f;
    }
    return g;
}

}  // namespace syn
