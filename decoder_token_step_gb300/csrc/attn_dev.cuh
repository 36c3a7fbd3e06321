// attn_dev.cuh -- split-K decode attention over the KV cache as device functions, used by the
// decode attention kernel (k_attn.cu) and the allocation-free entry point (attn_static.cu).
//
// `a = attention(q, k, v)` of "Local inference and architectures" (synsema.dev, section "The
// format"): for every query row at absolute position p and every query head h, with KV head
// g = h / (n_head / n_head_kv) (grouped-query sharing),
//     a_h = sum_t softmax_t(q_h . K_t / sqrt(hd)) V_t,  t in [lo, p],
// lo = 0 on global layers and p - window + 1 on sliding-window layers (window read from the GGUF
// metadata, "Rules"). The cache was appended to before this code runs ("Execution contract",
// section "Memory lifecycle / KV cache").
//
// Decode reads the whole cache of a layer once per step, so this is HBM-bound. One work item is one
// KV head for all the query heads that share it (K and V are read once per group, not once per
// query head) over one contiguous slice of the allowed keys. The slice count is fixed at launch (or
// derived on the device from the position) and the slice length is derived on the device from the
// current position, so a captured decode graph stays valid as the context grows.
//
// The kernels that use these functions stream K and V through a shared-memory ring filled by bulk
// copies; each consumer warp takes KB keys
// of a ring stage, lane l holding head-dimension elements l*EL .. l*EL+EL-1 of each row:
//   * per lane partial dot products for the KB keys x G heads are reduced with a warp
//     reduce-scatter (31 shuffles for 32 values), leaving one (key, head) score per lane;
//   * the online softmax (running max and sum per head) is kept per lane for its head;
//   * every lane accumulates the output of all G heads for its slice of the head dimension.
// Warps then merge in shared memory, and the last item of a (row, KV head) to finish merges the
// slices with their log-sum-exp weights (a completion counter; no CTA ever waits on another).
// All arithmetic is f32.
#pragma once

#include <cfloat>

#include "device_common.cuh"

namespace syn {

constexpr int kAttnWarps = 8;
constexpr int kAttnThreads = kAttnWarps * 32;

SYN_DEV void prefetch_l2(const void *ptr, unsigned bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(ptr), "r"(bytes) : "memory");
}

// Lane l ends with the warp-wide sum of v[l] (v has 32 entries per lane).
SYN_DEV float reduce_scatter32(float (&v)[32], int lane) {
#pragma unroll
    for (int half = 16; half >= 1; half >>= 1) {
        const bool up = lane & half;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float send = up ? v[i] : v[i + half];
            const float keep = up ? v[i + half] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, half);
        }
    }
    return v[0];
}

// vector load through L2 only (the data was written by an earlier kernel of the step)
template <int N> SYN_DEV void load_row(float (&dst)[N], const float *src) {
    if constexpr (N == 2) {
        const float2 a = __ldcg(reinterpret_cast<const float2 *>(src));
        dst[0] = a.x; dst[1] = a.y;
    } else {
#pragma unroll
        for (int i = 0; i < N; i += 4) {
            const float4 a = __ldcg(reinterpret_cast<const float4 *>(src + i));
            dst[i] = a.x; dst[i + 1] = a.y; dst[i + 2] = a.z; dst[i + 3] = a.w;
        }
    }
}

// Key slice [start, end) of work item (split, row). The position is fixed before a step's kernels
// run (it lives in device state written before the step), so the range is known early.
// Key slice `split` of query row `row` (keys [start, end), end exclusive) and the number of slices S
// in use at this step: about two ring stages of TK keys per slice or more, at most p.splits, so
// that short contexts and sliding windows run few work items and merge few partial results (the
// launch has p.splits items; those with split >= S have no keys and leave at once).
template <int TK>
SYN_DEV void attn_range(const AttnParams &p, int split, int row, int &pos, int &start, int &end, int &S) {
    pos = p.state->pos + row;
    const int lo = p.window > 0 ? max(0, pos - p.window + 1) : 0;
    const int len = pos - lo + 1;
    S = max(1, min(p.splits, (len + 2 * TK - 1) / (2 * TK)));
    const int chunk = (len + S - 1) / S;
    start = lo + split * chunk;
    end = split < S ? min(pos + 1, start + chunk) : start;  // exclusive
}

// EL consecutive cache elements of a shared-memory row, as f32 (EL = 2: one 8-byte load; else
// 16-byte loads; f16 rows are half as wide and widen exactly)
template <int EL> SYN_DEV void lds_row(float (&dst)[EL], const float *src) {
    if constexpr (EL == 2) {
        const float2 a = *reinterpret_cast<const float2 *>(src);
        dst[0] = a.x;
        dst[1] = a.y;
    } else {
#pragma unroll
        for (int e = 0; e < EL; e += 4) {
            const float4 a = *reinterpret_cast<const float4 *>(src + e);
            dst[e] = a.x; dst[e + 1] = a.y; dst[e + 2] = a.z; dst[e + 3] = a.w;
        }
    }
}
template <int EL> SYN_DEV void lds_row(float (&dst)[EL], const __half *src) {
    if constexpr (EL == 2) {
        const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(src));
        dst[0] = a.x;
        dst[1] = a.y;
    } else {
#pragma unroll
        for (int e = 0; e < EL; e += 4) {
            const uint2 w = *reinterpret_cast<const uint2 *>(src + e);
            const float2 a = __half22float2(*reinterpret_cast<const __half2 *>(&w.x));
            const float2 b = __half22float2(*reinterpret_cast<const __half2 *>(&w.y));
            dst[e] = a.x; dst[e + 1] = a.y; dst[e + 2] = b.x; dst[e + 3] = b.y;
        }
    }
}
SYN_DEV void st_kv(float *p, float v) { *p = v; }
SYN_DEV void st_kv(__half *p, float v) { *p = __float2half_rn(v); }

// Shared memory the compute part needs (bytes).
template <int HD, int GP> constexpr size_t attn_smem_bytes() {
    return (size_t)(2 * kAttnWarps * GP + kAttnWarps * GP * HD + GP * 64 + 4) * sizeof(float);
}

template <int HD, int GP> struct AttnShape {
    static constexpr int EL = HD / 32;                                        // head-dim elements per lane
    static constexpr int KB = (32 / GP) < (32 / EL) ? (32 / GP) : (32 / EL);  // keys per warp step
};

// This lane's slice of the G query heads of KV head g (zero for the padding heads).
template <int HD, int GP>
SYN_DEV void attn_load_q(const AttnParams &p, int g, int row, float (&q)[GP][HD / 32]) {
    constexpr int EL = HD / 32;
    const int G = p.n_head / p.n_kv, lane = threadIdx.x & 31;
#pragma unroll
    for (int h = 0; h < GP; ++h) {
        if (h < G) load_row<EL>(q[h], p.q + (size_t)row * p.ldq + (size_t)(g * G + h) * HD + lane * EL);
        else {
#pragma unroll
            for (int e = 0; e < EL; ++e) q[h][e] = 0.f;
        }
    }
}

// One warp step over nk (<= KB) keys whose rows this lane holds in kr: scores for every (key, head)
// pair, online-softmax update of the per-head running max m_run and sum l_run (kept by the lanes
// that own a head after the reduce-scatter), and accumulation of the output slices o. The value
// rows are fetched by vrow(j, v) one key at a time, after the scores (fewer live registers).
template <int HD, int GP, class VRow>
SYN_DEV void attn_step_v(const float (&q)[GP][HD / 32], const float (&kr)[AttnShape<HD, GP>::KB][HD / 32], VRow &&vrow,
                         int nk, int G, float scale, float &m_run, float &l_run, float (&o)[GP][HD / 32]) {
    constexpr int EL = HD / 32, KB = AttnShape<HD, GP>::KB;
    const int lane = threadIdx.x & 31;
    const int my_h = lane % GP;      // head of the (key, head) score this lane owns after reducing
    // partial scores, value index j * GP + h
    float sc[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) sc[i] = 0.f;
#pragma unroll
    for (int j = 0; j < KB; ++j)
#pragma unroll
        for (int h = 0; h < GP; ++h) {
            if constexpr (EL % 2 == 0) {
                // packed f32x2 products of element pairs, one add of the two halves at the end
                float2 s2 = make_float2(0.f, 0.f);
#pragma unroll
                for (int e = 0; e < EL; e += 2)
                    s2 = __ffma2_rn(make_float2(q[h][e], q[h][e + 1]), make_float2(kr[j][e], kr[j][e + 1]), s2);
                sc[j * GP + h] = s2.x + s2.y;
            } else {
                float s = 0.f;
#pragma unroll
                for (int e = 0; e < EL; ++e) s = fmaf(q[h][e], kr[j][e], s);
                sc[j * GP + h] = s;
            }
        }
    float s = reduce_scatter32(sc, lane) * scale;
    const int my_j = lane / GP;
    const bool valid = my_j < nk && my_h < G;
    if (!valid) s = -FLT_MAX;
    // per-head max and sum over the group's keys (lanes sharing my_h)
    float mx = s;
#pragma unroll
    for (int off = GP; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    const float m_new = fmaxf(m_run, mx);
    const float pr = valid ? expf(s - m_new) : 0.f;
    float ps = pr;
#pragma unroll
    for (int off = GP; off < 32; off <<= 1) ps += __shfl_xor_sync(0xffffffffu, ps, off);
    const float corr = expf(m_run - m_new);
    l_run = l_run * corr + ps;
    m_run = m_new;
    // rescale and accumulate every head's output slice
#pragma unroll
    for (int h = 0; h < GP; ++h) {
        const float c = __shfl_sync(0xffffffffu, corr, h);
#pragma unroll
        for (int e = 0; e < EL; ++e) o[h][e] *= c;
    }
#pragma unroll
    for (int j = 0; j < KB; ++j) {
        float vj[EL];
        vrow(j, vj);
#pragma unroll
        for (int h = 0; h < GP; ++h) {
            const float pj = __shfl_sync(0xffffffffu, pr, j * GP + h);
            if constexpr (EL % 2 == 0) {
#pragma unroll
                for (int e = 0; e < EL; e += 2) {
                    const float2 r2 = __ffma2_rn(make_float2(pj, pj), make_float2(vj[e], vj[e + 1]),
                                                 make_float2(o[h][e], o[h][e + 1]));
                    o[h][e] = r2.x;
                    o[h][e + 1] = r2.y;
                }
            } else {
#pragma unroll
                for (int e = 0; e < EL; ++e) o[h][e] = fmaf(pj, vj[e], o[h][e]);
            }
        }
    }
}

// attn_step with the value rows in registers
template <int HD, int GP>
SYN_DEV void attn_step(const float (&q)[GP][HD / 32], const float (&kr)[AttnShape<HD, GP>::KB][HD / 32],
                       const float (&vr)[AttnShape<HD, GP>::KB][HD / 32], int nk, int G, float scale, float &m_run,
                       float &l_run, float (&o)[GP][HD / 32]) {
    attn_step_v<HD, GP>(q, kr, [&](int j, float (&v)[HD / 32]) {
#pragma unroll
        for (int e = 0; e < HD / 32; ++e) v[e] = vr[j][e];
    }, nk, G, scale, m_run, l_run, o);
}

// Merge the kAttnWarps warps of this work item in shared memory and publish the slice's partial
// result; the last item of a (row, KV head) to finish merges all `splits` slices in use at this step
// (splits <= p.splits <= 64). Run by the first
// kAttnThreads threads of the block; `sync` is a barrier over exactly those threads.
template <int HD, int GP, class Sync>
SYN_DEV void attn_finish(const AttnParams &p, int splits, int g, int split, int row, float *smem, float m_run, float l_run,
                         const float (&o)[GP][HD / 32], Sync &&sync) {
    constexpr int EL = HD / 32;
    const int G = p.n_head / p.n_kv;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float (*wm)[GP] = reinterpret_cast<float (*)[GP]>(smem);
    float (*wl)[GP] = reinterpret_cast<float (*)[GP]>(smem + kAttnWarps * GP);
    float (*wo)[GP][HD] = reinterpret_cast<float (*)[GP][HD]>(smem + 2 * kAttnWarps * GP);
    float (*sw)[64] = reinterpret_cast<float (*)[64]>(smem + 2 * kAttnWarps * GP + kAttnWarps * GP * HD);
    int *last_flag = reinterpret_cast<int *>(smem + 2 * kAttnWarps * GP + kAttnWarps * GP * HD + GP * 64);
    if (lane < GP) {
        wm[warp][lane] = m_run;
        wl[warp][lane] = l_run;
    }
#pragma unroll
    for (int h = 0; h < GP; ++h)
#pragma unroll
        for (int e = 0; e < EL; ++e) wo[warp][h][lane * EL + e] = o[h][e];
    sync();
    // record per head: o[HD] (unnormalised), m, l, pad. The region of a (row, KV head) holds
    // p.splits records per head; this step uses the first `splits` (rows may use different counts)
    float *part = p.part + (((size_t)row * p.n_head + (size_t)g * G) * p.splits) * (HD + 4);
    const bool single = splits == 1;
    for (int idx = threadIdx.x; idx < G * HD; idx += kAttnThreads) {
        const int h = idx / HD, d = idx % HD;
        float M = -FLT_MAX;
#pragma unroll
        for (int w = 0; w < kAttnWarps; ++w) M = fmaxf(M, wm[w][h]);
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < kAttnWarps; ++w) {
            const float f = wl[w][h] > 0.f ? expf(wm[w][h] - M) : 0.f;
            L += f * wl[w][h];
            O += f * wo[w][h][d];
        }
        if (single) {
            p.out[(size_t)row * p.ldo + (size_t)(g * G + h) * HD + d] = O / L;
        } else {
            float *rec = part + ((size_t)h * splits + split) * (HD + 4);
            rec[d] = O;
            if (d == 0) {
                rec[HD] = L > 0.f ? M : -FLT_MAX;
                rec[HD + 1] = L;
            }
        }
    }
    if (single) {
        sync();  // the shared scratch is reused by whatever runs next in this CTA
        return;
    }

    // ---- the last CTA of this (row, KV head) merges all slices
    __threadfence();
    sync();
    if (threadIdx.x == 0) {
        unsigned *ctr = p.counters + (size_t)row * p.n_kv + g;
        const bool last = atomicAdd(ctr, 1u) == (unsigned)splits - 1;
        if (last) *ctr = 0;  // ready for the next step (every CTA of this launch has arrived)
        *last_flag = last;
    }
    sync();
    if (!*last_flag) return;
    __threadfence();
    for (int h = warp; h < G; h += kAttnWarps) {
        // weights exp(m_s - M) of every slice of head h; splits <= 64 on this path
        float M = -FLT_MAX;
        for (int s2 = lane; s2 < splits; s2 += 32) M = fmaxf(M, __ldcg(part + ((size_t)h * splits + s2) * (HD + 4) + HD));
        M = warp_max(M);
        for (int s2 = lane; s2 < splits; s2 += 32) {
            const float *rec = part + ((size_t)h * splits + s2) * (HD + 4);
            const float l2 = __ldcg(rec + HD + 1);
            sw[h][s2] = l2 > 0.f ? expf(__ldcg(rec + HD) - M) : 0.f;
        }
    }
    sync();
    for (int idx = threadIdx.x; idx < G * HD; idx += kAttnThreads) {
        const int h = idx / HD, d = idx % HD;
        // the slices' records are independent L2 reads: eight in flight at a time, summed in order
        float L = 0.f, O = 0.f;
        for (int s0 = 0; s0 < splits; s0 += 8) {
            float lv[8], ov[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float *rec = part + ((size_t)h * splits + min(s0 + j, splits - 1)) * (HD + 4);
                lv[j] = __ldcg(rec + HD + 1);
                ov[j] = __ldcg(rec + d);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (s0 + j < splits) {
                    const float w = sw[h][s0 + j];
                    L = fmaf(w, lv[j], L);
                    O = fmaf(w, ov[j], O);
                }
            }
        }
        p.out[(size_t)row * p.ldo + (size_t)(g * G + h) * HD + d] = O / L;
    }
    sync();
}


}  // namespace syn
