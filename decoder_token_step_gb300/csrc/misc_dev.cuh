// misc_dev.cuh -- the small ops of the decoder step as device functions, used by the kernels of
// k_misc.cu, k_attn.cu and attn_static.cu: embed, RMSNorm, the per-head
// transforms before attention (add_bias, norm_heads, rope, KV append), elementwise ops and the greedy
// argmax. Ops of "Local inference and architectures" (synsema.dev, section "The operations"); each
// works on `rows` rows so the same code serves decode (1 row) and bulk prefill, and spreads its work
// over `ncta` CTAs. Activations written by other CTAs are read through L2 only (__ldcg).
#pragma once

#include <cfloat>

#include "device_common.cuh"

namespace syn {

// The threads that run an op inside a CTA (the whole block): index, count and barrier.
struct BlockThreads {
    static SYN_DEV int tid() { return threadIdx.x; }
    static SYN_DEV int n() { return blockDim.x; }
    static SYN_DEV void sync() { __syncthreads(); }
};

template <class T = BlockThreads> SYN_DEV float block_sum(float v, float *red) {
    const int lane = T::tid() & 31, warp = T::tid() >> 5, nw = (T::n() + 31) / 32;
    v = warp_sum(v);
    T::sync();
    if (lane == 0) red[warp] = v;
    T::sync();
    float t = 0.f;
    for (int i = 0; i < nw; ++i) t += red[i];
    return t;
}

// x[r] = dequant(E[tokens[r]]) * scale   (`embed`, optionally with a folded `scale` step)
template <class T = BlockThreads> SYN_DEV void embed_cta(const EmbedParams &p, int cta, int ncta) {
    const int64_t total = (int64_t)p.n * p.E.K;
    for (int64_t i = (int64_t)cta * T::n() + T::tid(); i < total; i += (int64_t)ncta * T::n()) {
        const int r = (int)(i / p.E.K);
        const int64_t k = i % p.E.K;
        int tok = p.tokens[r];
        if (tok < 0 || tok >= p.E.N) {
            if (k == 0) atomicOr(&p.state->err, ERR_TOKEN_RANGE);
            tok = -1;
        }
        const float v = tok < 0 ? 0.f : dequant_one(p.E, tok, k);
        p.out[(size_t)r * p.E.K + k] = p.scale == 1.f ? v : v * p.scale;
    }
}

// y = x / sqrt(mean(x^2) + eps) * w, one CTA per row; or residual += that (post-branch norm).
// Four floats per access when the width, the row stride and the pointers allow it.
template <class T = BlockThreads> SYN_DEV void rms_cta(const RmsParams &p, int cta, int ncta, float *red) {
    const bool vec = p.width % 4 == 0 && p.ld % 4 == 0 &&
                     ((reinterpret_cast<uintptr_t>(p.x) | reinterpret_cast<uintptr_t>(p.w) | reinterpret_cast<uintptr_t>(p.y) |
                       reinterpret_cast<uintptr_t>(p.residual)) & 15) == 0;
    if (vec) {
        const int w4 = p.width / 4;
        const float4 *w = reinterpret_cast<const float4 *>(p.w);
        for (int r = cta; r < p.rows; r += ncta) {
            const float4 *x = reinterpret_cast<const float4 *>(p.x + (size_t)r * p.ld);
            float ss = 0.f;
            for (int i = T::tid(); i < w4; i += T::n()) {
                const float4 v = __ldcg(x + i);
                ss = fmaf(v.x, v.x, ss);
                ss = fmaf(v.y, v.y, ss);
                ss = fmaf(v.z, v.z, ss);
                ss = fmaf(v.w, v.w, ss);
            }
            ss = block_sum<T>(ss, red);
            const float inv = 1.f / sqrtf(ss / (float)p.width + p.eps);
            float4 *out = reinterpret_cast<float4 *>((p.residual ? p.residual : p.y) + (size_t)r * p.ld);
            for (int i = T::tid(); i < w4; i += T::n()) {
                const float4 v = __ldcg(x + i), g = w[i];
                float4 y = make_float4(v.x * inv * g.x, v.y * inv * g.y, v.z * inv * g.z, v.w * inv * g.w);
                if (p.residual) {
                    const float4 o = __ldcg(out + i);
                    y = make_float4(o.x + y.x, o.y + y.y, o.z + y.z, o.w + y.w);
                }
                out[i] = y;
            }
            T::sync();
        }
        return;
    }
    for (int r = cta; r < p.rows; r += ncta) {
        const float *x = p.x + (size_t)r * p.ld;
        float ss = 0.f;
        for (int i = T::tid(); i < p.width; i += T::n()) {
            const float v = __ldcg(x + i);
            ss = fmaf(v, v, ss);
        }
        ss = block_sum<T>(ss, red);
        const float inv = 1.f / sqrtf(ss / (float)p.width + p.eps);
        if (p.residual) {
            float *res = p.residual + (size_t)r * p.ld;
            for (int i = T::tid(); i < p.width; i += T::n()) res[i] = __ldcg(res + i) + __ldcg(x + i) * inv * p.w[i];
        } else {
            float *y = p.y + (size_t)r * p.ld;
            for (int i = T::tid(); i < p.width; i += T::n()) y[i] = __ldcg(x + i) * inv * p.w[i];
        }
        T::sync();
    }
}

SYN_DEV float elt_one(const EltParams &p, float a, size_t o, int c) {
    switch (p.op) {
    case ELT_ACT: return apply_act(p.act, a);
    case ELT_MUL: return a * __ldcg(p.b + o);
    case ELT_ADD: return a + __ldcg(p.b + o);
    case ELT_SCALE: return a * p.c;
    case ELT_BIAS: return a + p.b[c];
    case ELT_ACT_MUL: return apply_act(p.act, a) * __ldcg(p.b + o);
    default: return a;
    }
}

// y = op(a[, b]) over rows x width (row stride ld). Four consecutive elements per step when the
// width, the stride and the pointers allow 16-byte accesses; one otherwise.
template <class T = BlockThreads> SYN_DEV void elt_cta(const EltParams &p, int cta, int ncta) {
    const bool vec = (p.width % 4 == 0) && (p.ld % 4 == 0) && ((reinterpret_cast<uintptr_t>(p.a) | reinterpret_cast<uintptr_t>(p.y) |
                                                                 reinterpret_cast<uintptr_t>(p.b)) & 15) == 0;
    if (vec) {
        const int w4 = p.width / 4;
        const int64_t n = (int64_t)p.rows * w4;
        for (int64_t i = (int64_t)cta * T::n() + T::tid(); i < n; i += (int64_t)ncta * T::n()) {
            const int r = (int)(i / w4), c = (int)(i - (int64_t)r * w4) * 4;
            const size_t o = (size_t)r * p.ld + c;
            const float4 a = __ldcg(reinterpret_cast<const float4 *>(p.a + o));
            float4 v;
            v.x = elt_one(p, a.x, o, c);
            v.y = elt_one(p, a.y, o + 1, c + 1);
            v.z = elt_one(p, a.z, o + 2, c + 2);
            v.w = elt_one(p, a.w, o + 3, c + 3);
            *reinterpret_cast<float4 *>(p.y + o) = v;
        }
        return;
    }
    const int64_t n = (int64_t)p.rows * p.width;
    for (int64_t i = (int64_t)cta * T::n() + T::tid(); i < n; i += (int64_t)ncta * T::n()) {
        const int64_t r = i / p.width, c = i % p.width;
        const size_t o = (size_t)r * p.ld + c;
        p.y[o] = elt_one(p, __ldcg(p.a + o), o, (int)c);
    }
}

// The per-head transforms of one head held by one warp, lane l holding elements l*PL .. l*PL+PL-1
// (PL = HD / 32), in the archdef's order: bias (add_bias), RMS norm over the head (norm_heads,
// weight w of HD floats), rotary embedding at the row's position (rope; cs = the position's HD/2
// (cos, sin) pairs). bias / w null and do_rope 0 skip a step.
template <int HD>
SYN_DEV void head_transform(float (&v)[HD / 32], const float *bias, const float *w, int do_rope, const float2 *cs,
                            int adjacent, float eps) {
    constexpr int PL = HD / 32;
    const int lane = threadIdx.x & 31;
    if (bias) {
#pragma unroll
        for (int i = 0; i < PL; ++i) v[i] += bias[lane * PL + i];
    }
    if (w) {
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < PL; ++i) ss = fmaf(v[i], v[i], ss);
        ss = warp_sum(ss);
        const float inv = 1.f / sqrtf(ss / (float)HD + eps);
#pragma unroll
        for (int i = 0; i < PL; ++i) v[i] = v[i] * inv * w[lane * PL + i];
    }
    if (do_rope) {
        if (adjacent) {
            // pairs (2j, 2j+1) are both in this lane
#pragma unroll
            for (int i = 0; i < PL; i += 2) {
                const int j = (lane * PL + i) / 2;
                const float2 c = cs[j];
                const float a = v[i], b = v[i + 1];
                v[i] = a * c.x - b * c.y;
                v[i + 1] = a * c.y + b * c.x;
            }
        } else {
            // pairs (j, j + HD/2): the partner element lives in lane ^ 16
#pragma unroll
            for (int i = 0; i < PL; ++i) {
                const float other = __shfl_xor_sync(0xffffffffu, v[i], 16);
                const int e = lane * PL + i;
                const bool first = e < HD / 2;
                const float2 c = cs[first ? e : e - HD / 2];
                // first half: a*cos - b*sin with b the partner; second half: a*sin + b*cos with a the partner
                v[i] = first ? v[i] * c.x - other * c.y : other * c.y + v[i] * c.x;
            }
        }
    }
}

// The same steps with the constants already in registers (loaded before the kernel waited for the
// one that wrote v): b and w when has_b / has_w, and c[i] the rope (cos, sin) of this lane's element
// i -- for adjacent pairs, the pair's entry at both of its elements.
template <int HD>
SYN_DEV void head_transform_r(float (&v)[HD / 32], bool has_b, const float (&b)[HD / 32], bool has_w,
                              const float (&w)[HD / 32], int do_rope, const float2 (&c)[HD / 32], int adjacent,
                              float eps) {
    constexpr int PL = HD / 32;
    const int lane = threadIdx.x & 31;
    if (has_b) {
#pragma unroll
        for (int i = 0; i < PL; ++i) v[i] += b[i];
    }
    if (has_w) {
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < PL; ++i) ss = fmaf(v[i], v[i], ss);
        ss = warp_sum(ss);
        const float inv = 1.f / sqrtf(ss / (float)HD + eps);
#pragma unroll
        for (int i = 0; i < PL; ++i) v[i] = v[i] * inv * w[i];
    }
    if (do_rope) {
        if (adjacent) {
#pragma unroll
            for (int i = 0; i < PL; i += 2) {
                const float a = v[i], bb = v[i + 1];
                v[i] = a * c[i].x - bb * c[i].y;
                v[i + 1] = a * c[i].y + bb * c[i].x;
            }
        } else {
#pragma unroll
            for (int i = 0; i < PL; ++i) {
                const float other = __shfl_xor_sync(0xffffffffu, v[i], 16);
                const bool first = lane * PL + i < HD / 2;
                v[i] = first ? v[i] * c[i].x - other * c[i].y : other * c[i].y + v[i] * c[i].x;
            }
        }
    }
}
// This lane's rope factors for head_transform_r, position pos.
template <int HD>
SYN_DEV void rope_factors(float2 (&c)[HD / 32], const float2 *rope_cs, int pos, int adjacent) {
    constexpr int PL = HD / 32;
    const int lane = threadIdx.x & 31;
    const float2 *cs = rope_cs + (size_t)pos * (HD / 2);
#pragma unroll
    for (int i = 0; i < PL; ++i) {
        const int e = lane * PL + i;
        c[i] = cs[adjacent ? e / 2 : (e < HD / 2 ? e : e - HD / 2)];
    }
}

// One warp per (row, head): q heads first, then k heads. Steps in order: bias, norm_heads, rope;
// k heads (and the matching v rows) are then written into the cache at position pos + row.
template <int HD>
SYN_DEV void heads_warp(const HeadsParams &p, int warp_global) {
    constexpr int PL = HD / 32;                     // elements per lane (consecutive)
    const int lane = threadIdx.x & 31;
    const int per_row = p.nq + p.nk;
    const int row = warp_global / per_row, h = warp_global % per_row;
    const bool is_q = h < p.nq;
    const int hh = is_q ? h : h - p.nq;
    float *src = is_q ? p.q + (size_t)row * p.ldq + (size_t)hh * HD : p.k + (size_t)row * p.ldk + (size_t)hh * HD;
    const float *bias = is_q ? p.bq : p.bk;
    const int pos = p.state->pos + row;

    float v[PL];
#pragma unroll
    for (int i = 0; i < PL; ++i) v[i] = __ldcg(src + lane * PL + i);
    head_transform<HD>(v, bias ? bias + (size_t)hh * HD : nullptr, is_q ? p.wq : p.wk, is_q ? p.rope_q : p.rope_k,
                       p.rope_cs + (size_t)pos * (HD / 2), p.rope_adjacent, p.eps);
    if (!is_q && p.kcache) {
        const size_t at = ((size_t)hh * p.max_ctx + pos) * HD + lane * PL;
        const float *vs = p.v + (size_t)row * p.ldv + (size_t)hh * HD;
#pragma unroll
        for (int i = 0; i < PL; ++i) {
            float vv = __ldcg(vs + lane * PL + i);
            if (p.bv) vv += p.bv[(size_t)hh * HD + lane * PL + i];
            if (p.kv_f16) {
                static_cast<__half *>(p.kcache)[at + i] = __float2half_rn(v[i]);
                static_cast<__half *>(p.vcache)[at + i] = __float2half_rn(vv);
            } else {
                static_cast<float *>(p.kcache)[at + i] = v[i];
                static_cast<float *>(p.vcache)[at + i] = vv;
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < PL; ++i) src[lane * PL + i] = v[i];
    }
}

// the heads of all rows, one warp each, spread over the CTAs
template <class T = BlockThreads> SYN_DEV void heads_cta(const HeadsParams &p, int cta, int ncta) {
    const int warps = T::n() / 32;
    const int total = (p.nq + p.nk) * p.rows;
    for (int w = cta * warps + (T::tid() >> 5); w < total; w += ncta * warps) {
        switch (p.hd) {
        case 64: heads_warp<64>(p, w); break;
        case 128: heads_warp<128>(p, w); break;
        case 256: heads_warp<256>(p, w); break;
        }
    }
}

// greedy argmax: largest value, lowest index on ties; NaN never wins
SYN_DEV bool better(float v, int i, float bv, int bi) { return v > bv || (v == bv && i < bi); }

template <class T = BlockThreads>
SYN_DEV void argmax_cta(const ArgmaxParams &p, int cta, int ncta, float *sv, int *si, int *last_flag) {
    float bv = -FLT_MAX;
    int bi = 0x7fffffff;
    for (int i = cta * T::n() + T::tid(); i < p.n; i += ncta * T::n()) {
        const float v = __ldcg(p.x + i);
        if (better(v, i, bv, bi)) { bv = v; bi = i; }
    }
    const int lane = T::tid() & 31, warp = T::tid() >> 5, nw = T::n() / 32;
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
    }
    if (lane == 0) { sv[warp] = bv; si[warp] = bi; }
    T::sync();
    if (T::tid() == 0) {
        for (int w = 1; w < nw; ++w)
            if (better(sv[w], si[w], bv, bi)) { bv = sv[w]; bi = si[w]; }
        p.part_v[cta] = bv;
        p.part_i[cta] = bi;
        __threadfence();
        *last_flag = atomicAdd(p.counter, 1u) == (unsigned)ncta - 1;
    }
    T::sync();
    if (*last_flag && T::tid() == 0) {
        // the last CTA to finish reduces the per-CTA results (no CTA waits on another)
        __threadfence();
        float v = -FLT_MAX;
        int idx = 0x7fffffff;
        for (int b = 0; b < ncta; ++b) {
            const float pv = ((volatile float *)p.part_v)[b];
            const int pi = ((volatile int *)p.part_i)[b];
            if (better(pv, pi, v, idx)) { v = pv; idx = pi; }
        }
        p.state->argmax = idx;
        *p.counter = 0;
        if (p.advance) p.state->pos += p.state->n;
    }
    T::sync();
}


}  // namespace syn
