// k_attn.cu -- attention over the KV cache (split-K "flash decode").
//
// `a = attention(q, k, v)` of "Local inference and architectures" (synsema.dev, section "The
// format"): for every query row at absolute position p and every query head h, with KV head
// g = h / (n_head / n_head_kv) (grouped-query sharing),
//     a_h = sum_t softmax_t(q_h . K_t / sqrt(hd)) V_t,  t in [lo, p],
// lo = 0 on global layers and p - window + 1 on sliding-window layers (window read from the GGUF
// metadata, "Rules"). The cache was appended to before this kernel runs ("Execution contract",
// section "Memory lifecycle / KV cache").
//
// Decode reads the whole cache of a layer once per step, so this is HBM-bound. One CTA handles one
// KV head for all the query heads that share it (K and V are read once per group, not once per
// query head) over one contiguous slice of the allowed keys. The slice count is fixed at launch
// and the slice length is derived on the device from the current position, so a captured decode
// graph stays valid as the context grows.
//
// Inside a CTA every warp streams its own groups of KB keys straight from HBM into registers
// (coalesced: a key row per warp-wide vector load), with no shared-memory staging and no
// block-wide barrier per tile:
//   * per lane partial dot products for the KB keys x G heads are reduced with a warp
//     reduce-scatter (31 shuffles for 32 values), leaving one (key, head) score per lane;
//   * the online softmax (running max and sum per head) is kept per lane for its head;
//   * every lane accumulates the output of all G heads for its slice of the head dimension.
// Warps then merge in shared memory, and the last CTA of a (row, KV head) to finish merges the
// slices with their log-sum-exp weights (a completion counter; no CTA ever waits on another).
// All arithmetic is f32.
#include <cfloat>

#include "device_common.cuh"

namespace syn {

namespace {

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

// HD: head dimension; GP: query heads per KV head rounded up to a power of two.
template <int HD, int GP>
__global__ void __launch_bounds__(kAttnThreads) k_attn(const AttnParams p) {
    constexpr int EL = HD / 32;                                  // head-dim elements per lane
    constexpr int KB = (32 / GP) < (32 / EL) ? (32 / GP) : (32 / EL);  // keys per warp step
    const int g = blockIdx.x, split = blockIdx.y, row = blockIdx.z;
    const int G = p.n_head / p.n_kv;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const float *Kg = p.kcache + (size_t)g * p.max_ctx * HD;
    const float *Vg = p.vcache + (size_t)g * p.max_ctx * HD;

    // the position is fixed before this step's kernels run, so the key range is known early
    const int pos = p.state->pos + row;
    const int lo = p.window > 0 ? max(0, pos - p.window + 1) : 0;
    const int len = pos - lo + 1;
    const int chunk = (len + p.splits - 1) / p.splits;
    const int start = lo + split * chunk;
    const int end = min(pos + 1, start + chunk);  // exclusive
    // keys before pos were written by earlier steps: start pulling them into L2 now
    if (threadIdx.x == 0 && start < min(end, pos)) {
        const unsigned bytes = (unsigned)(min(end, pos) - start) * HD * 4u;
        prefetch_l2(Kg + (size_t)start * HD, bytes);
        prefetch_l2(Vg + (size_t)start * HD, bytes);
    }
    pdl_launch_dependents();
    pdl_wait();

    // this lane's slice of the G query heads
    float q[GP][EL];
#pragma unroll
    for (int h = 0; h < GP; ++h) {
        if (h < G) load_row<EL>(q[h], p.q + (size_t)row * p.ldq + (size_t)(g * G + h) * HD + lane * EL);
        else {
#pragma unroll
            for (int e = 0; e < EL; ++e) q[h][e] = 0.f;
        }
    }
    const float scale = 1.f / sqrtf((float)HD);
    const int my_h = lane % GP;      // head of the (key, head) score this lane owns after reducing
    float m_run = -FLT_MAX, l_run = 0.f;
    float o[GP][EL];
#pragma unroll
    for (int h = 0; h < GP; ++h)
#pragma unroll
        for (int e = 0; e < EL; ++e) o[h][e] = 0.f;

    for (int t0 = start + warp * KB; t0 < end; t0 += kAttnWarps * KB) {
        const int nk = min(KB, end - t0);
        float kr[KB][EL], vr[KB][EL];
#pragma unroll
        for (int j = 0; j < KB; ++j) {
            if (j < nk) {
                load_row<EL>(kr[j], Kg + (size_t)(t0 + j) * HD + lane * EL);
                load_row<EL>(vr[j], Vg + (size_t)(t0 + j) * HD + lane * EL);
            } else {
#pragma unroll
                for (int e = 0; e < EL; ++e) { kr[j][e] = 0.f; vr[j][e] = 0.f; }
            }
        }
        // partial scores, value index j * GP + h
        float sc[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) sc[i] = 0.f;
#pragma unroll
        for (int j = 0; j < KB; ++j)
#pragma unroll
            for (int h = 0; h < GP; ++h) {
                float s = 0.f;
#pragma unroll
                for (int e = 0; e < EL; ++e) s = fmaf(q[h][e], kr[j][e], s);
                sc[j * GP + h] = s;
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
        for (int j = 0; j < KB; ++j)
#pragma unroll
            for (int h = 0; h < GP; ++h) {
                const float pj = __shfl_sync(0xffffffffu, pr, j * GP + h);
#pragma unroll
                for (int e = 0; e < EL; ++e) o[h][e] = fmaf(pj, vr[j][e], o[h][e]);
            }
    }

    // ---- merge the warps of this CTA (shared memory), then publish the slice's partial result
    __shared__ float wm[kAttnWarps][GP], wl[kAttnWarps][GP];
    __shared__ __align__(16) float wo[kAttnWarps][GP][HD];
    if (lane < GP) {
        wm[warp][lane] = m_run;
        wl[warp][lane] = l_run;
    }
#pragma unroll
    for (int h = 0; h < GP; ++h)
#pragma unroll
        for (int e = 0; e < EL; ++e) wo[warp][h][lane * EL + e] = o[h][e];
    __syncthreads();
    // record per head: o[HD] (unnormalised), m, l, pad
    float *part = p.part + (((size_t)row * p.n_head + (size_t)g * G) * p.splits) * (HD + 4);
    const bool single = p.splits == 1;
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
            float *rec = part + ((size_t)h * p.splits + split) * (HD + 4);
            rec[d] = O;
            if (d == 0) {
                rec[HD] = L > 0.f ? M : -FLT_MAX;
                rec[HD + 1] = L;
            }
        }
    }
    if (single) return;

    // ---- the last CTA of this (row, KV head) merges all slices
    __shared__ bool last;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned *ctr = p.counters + (size_t)row * p.n_kv + g;
        last = atomicAdd(ctr, 1u) == (unsigned)p.splits - 1;
        if (last) *ctr = 0;  // ready for the next step (every CTA of this launch has arrived)
    }
    __syncthreads();
    if (!last) return;
    __threadfence();
    __shared__ float sw[GP][64];
    for (int h = warp; h < G; h += kAttnWarps) {
        // weights exp(m_s - M) of every slice of head h; splits <= 64 on this path
        float M = -FLT_MAX;
        for (int s2 = lane; s2 < p.splits; s2 += 32) M = fmaxf(M, __ldcg(part + ((size_t)h * p.splits + s2) * (HD + 4) + HD));
        M = warp_max(M);
        for (int s2 = lane; s2 < p.splits; s2 += 32) {
            const float *rec = part + ((size_t)h * p.splits + s2) * (HD + 4);
            const float l2 = __ldcg(rec + HD + 1);
            sw[h][s2] = l2 > 0.f ? expf(__ldcg(rec + HD) - M) : 0.f;
        }
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < G * HD; idx += kAttnThreads) {
        const int h = idx / HD, d = idx % HD;
        float L = 0.f, O = 0.f;
        for (int s2 = 0; s2 < p.splits; ++s2) {
            const float *rec = part + ((size_t)h * p.splits + s2) * (HD + 4);
            const float w = sw[h][s2];
            L = fmaf(w, __ldcg(rec + HD + 1), L);
            O = fmaf(w, __ldcg(rec + d), O);
        }
        p.out[(size_t)row * p.ldo + (size_t)(g * G + h) * HD + d] = O / L;
    }
}

template <int HD, int GP> void launch_t(const AttnParams &p, cudaStream_t s, bool pdl) {
    if (pdl)
        launch_pdl(k_attn<HD, GP>, dim3(p.n_kv, p.splits, p.rows), dim3(kAttnThreads), 0, s, p);
    else
        k_attn<HD, GP><<<dim3(p.n_kv, p.splits, p.rows), kAttnThreads, 0, s>>>(p);
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
