// device_common.cuh -- small device helpers of the libsyn kernels (weight decoding, reductions,
// streaming loads). Internal to the CUDA sources.
#pragma once

#include <cuda_fp16.h>
#include <cstdint>

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

// Small integer codes to f32 without an int->float conversion instruction: a byte b placed in the
// low mantissa bits of 2^23 gives the float 2^23 + b exactly; subtracting 2^23 + offset leaves
// b - offset exactly (all values involved are integers below 2^24).
SYN_DEV float byte_to_float(uint32_t word, int which, float bias) {
    // which selects byte 0..3 of word; constant bytes come from 0x4B000000 (the float 2^23)
    const uint32_t sel = 0x7440u | (uint32_t)which;
    return __uint_as_float(__byte_perm(word, 0x4B000000u, sel)) - bias;
}

// Dot product of one 16-byte chunk of a row with the matching x values. `xs` points at the
// chunk's slot in shared memory laid out so that float4 number j of lane l sits at
// xs[j * 128 + l * 4] (lane-interleaved, conflict-free). Returns the f32 partial sum; for the
// quantised types the block scale is applied by the caller.
template <int WT> struct Chunk;

template <> struct Chunk<W_F32> {
    static constexpr int E = 4;  // elements per 16 bytes
    static SYN_DEV float dot(uint4 w, const float *xs) {
        float4 x = *reinterpret_cast<const float4 *>(xs);
        return __uint_as_float(w.x) * x.x + __uint_as_float(w.y) * x.y + __uint_as_float(w.z) * x.z +
               __uint_as_float(w.w) * x.w;
    }
};

template <> struct Chunk<W_F16> {
    static constexpr int E = 8;
    static SYN_DEV float dot(uint4 w, const float *xs) {
        float4 x0 = *reinterpret_cast<const float4 *>(xs);
        float4 x1 = *reinterpret_cast<const float4 *>(xs + 128);
        float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&w.x));
        float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&w.y));
        float2 c = __half22float2(*reinterpret_cast<const __half2 *>(&w.z));
        float2 d = __half22float2(*reinterpret_cast<const __half2 *>(&w.w));
        float s = a.x * x0.x;
        s = fmaf(a.y, x0.y, s);
        s = fmaf(b.x, x0.z, s);
        s = fmaf(b.y, x0.w, s);
        s = fmaf(c.x, x1.x, s);
        s = fmaf(c.y, x1.y, s);
        s = fmaf(d.x, x1.z, s);
        s = fmaf(d.y, x1.w, s);
        return s;
    }
};

// Q8_0: 16 signed codes; flip the sign bit to make them offset-binary, then decode with bias 128.
template <> struct Chunk<W_Q8_0> {
    static constexpr int E = 16;
    static SYN_DEV float dot4(uint32_t w, float4 x) {
        w ^= 0x80808080u;
        float s = byte_to_float(w, 0, 8388736.f) * x.x;
        s = fmaf(byte_to_float(w, 1, 8388736.f), x.y, s);
        s = fmaf(byte_to_float(w, 2, 8388736.f), x.z, s);
        s = fmaf(byte_to_float(w, 3, 8388736.f), x.w, s);
        return s;
    }
    static SYN_DEV float dot(uint4 w, const float *xs) {
        float s = dot4(w.x, *reinterpret_cast<const float4 *>(xs));
        s += dot4(w.y, *reinterpret_cast<const float4 *>(xs + 128));
        s += dot4(w.z, *reinterpret_cast<const float4 *>(xs + 256));
        s += dot4(w.w, *reinterpret_cast<const float4 *>(xs + 384));
        return s;
    }
};

// Q4_0: one whole 32-weight block per 16 bytes. Word i holds elements 4i..4i+3 in its low nibbles
// and 16+4i..16+4i+3 in its high nibbles; codes decode to code - 8.
template <> struct Chunk<W_Q4_0> {
    static constexpr int E = 32;
    static SYN_DEV float dot4(uint32_t nib, float4 x) {
        float s = byte_to_float(nib, 0, 8388616.f) * x.x;
        s = fmaf(byte_to_float(nib, 1, 8388616.f), x.y, s);
        s = fmaf(byte_to_float(nib, 2, 8388616.f), x.z, s);
        s = fmaf(byte_to_float(nib, 3, 8388616.f), x.w, s);
        return s;
    }
    static SYN_DEV float dot(uint4 w, const float *xs) {
        const uint32_t m = 0x0F0F0F0Fu;
        float s = dot4(w.x & m, *reinterpret_cast<const float4 *>(xs + 0 * 128));
        s += dot4(w.y & m, *reinterpret_cast<const float4 *>(xs + 1 * 128));
        s += dot4(w.z & m, *reinterpret_cast<const float4 *>(xs + 2 * 128));
        s += dot4(w.w & m, *reinterpret_cast<const float4 *>(xs + 3 * 128));
        s += dot4((w.x >> 4) & m, *reinterpret_cast<const float4 *>(xs + 4 * 128));
        s += dot4((w.y >> 4) & m, *reinterpret_cast<const float4 *>(xs + 5 * 128));
        s += dot4((w.z >> 4) & m, *reinterpret_cast<const float4 *>(xs + 6 * 128));
        s += dot4((w.w >> 4) & m, *reinterpret_cast<const float4 *>(xs + 7 * 128));
        return s;
    }
};

// Element e of the chunk of lane l in group g sits at this shared-memory offset (see Chunk).
template <int E> SYN_DEV int xs_offset(int g, int l, int e) { return g * 32 * E + (e >> 2) * 128 + l * 4 + (e & 3); }

// Dequantised value of element k of row `row` of W (f32; exact: d * code).
SYN_DEV float dequant_one(const DevMatrix &W, int64_t row, int64_t k) {
    const uint8_t *rp = reinterpret_cast<const uint8_t *>(W.codes) + (size_t)row * W.row_bytes;
    switch (W.wtype) {
    case W_F32: return reinterpret_cast<const float *>(rp)[k];
    case W_F16: return half_bits_to_float(reinterpret_cast<const uint16_t *>(rp)[k]);
    case W_Q8_0: {
        float d = half_bits_to_float(W.scales[(size_t)row * (W.K / 32) + k / 32]);
        return d * (float)(int8_t)rp[k];
    }
    case W_Q4_0: {
        float d = half_bits_to_float(W.scales[(size_t)row * (W.K / 32) + k / 32]);
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
