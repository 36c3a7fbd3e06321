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
// query head) over one contiguous slice of the allowed keys; the slice count is fixed at launch
// and the slice length is derived on the device from the current position, so a captured decode
// graph stays valid as the context grows. K/V tiles are staged in shared memory with cp.async
// (double-buffered); scores, the running max / sum and the output accumulators are f32. A second
// kernel merges the slices with their log-sum-exp weights.
#include <cfloat>

#include "device_common.cuh"

namespace syn {

namespace {

constexpr int kAttnThreads = 128;
constexpr int kMaxG = 8;             // query heads per KV head handled by one CTA

SYN_DEV void cp_async16(void *smem, const void *gmem) {
    unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem));
}
SYN_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;"); }
template <int N> SYN_DEV void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N)); }

// T keys of HD floats per tile: 16 KB per K tile and per V tile.
template <int HD> struct Tile { static constexpr int T = 4096 / HD; };

template <int HD>
__global__ void __launch_bounds__(kAttnThreads) k_attn_split(const AttnParams p) {
    constexpr int T = Tile<HD>::T;
    constexpr int V4 = HD / 4;                     // float4 per key row
    extern __shared__ __align__(16) float sm[];
    float *Ks = sm;                                // [2][T][HD]
    float *Vs = Ks + 2 * T * HD;                   // [2][T][HD]
    float *qs = Vs + 2 * T * HD;                   // [G][HD]
    float *ps = qs + kMaxG * HD;                   // [G][T] scores, then probabilities
    __shared__ float m_run[kMaxG], l_run[kMaxG], corr[kMaxG];

    const int g = blockIdx.x, split = blockIdx.y, row = blockIdx.z;
    const int G = p.n_head / p.n_kv;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int pos = p.state->pos + row;
    const int lo = p.window > 0 ? max(0, pos - p.window + 1) : 0;
    const int len = pos - lo + 1;
    const int chunk = (len + p.splits - 1) / p.splits;
    const int start = lo + split * chunk;
    const int end = min(pos + 1, start + chunk);   // exclusive
    const float scale = 1.f / sqrtf((float)HD);

    float *part = p.part + ((size_t)row * p.n_head + (size_t)g * G) * p.splits * (HD + 4);

    // load the G query heads of this group
    for (int i = tid; i < G * HD; i += kAttnThreads)
        qs[i] = p.q[(size_t)row * p.ldq + (size_t)g * G * HD + i];
    if (tid < kMaxG) { m_run[tid] = -FLT_MAX; l_run[tid] = 0.f; }

    constexpr int kSlots = (kMaxG * V4 + kAttnThreads - 1) / kAttnThreads;
    float4 acc[kSlots];
#pragma unroll
    for (int i = 0; i < kSlots; ++i) acc[i] = make_float4(0, 0, 0, 0);

    const float *Kg = p.kcache + (size_t)g * p.max_ctx * HD;
    const float *Vg = p.vcache + (size_t)g * p.max_ctx * HD;
    const int ntiles = start < end ? (end - start + T - 1) / T : 0;

    auto load_tile = [&](int t, int buf) {
        const int t0 = start + t * T;
        const int nk = min(T, end - t0);
        for (int i = tid; i < nk * V4; i += kAttnThreads) {
            cp_async16(Ks + (size_t)buf * T * HD + i * 4, Kg + (size_t)t0 * HD + i * 4);
            cp_async16(Vs + (size_t)buf * T * HD + i * 4, Vg + (size_t)t0 * HD + i * 4);
        }
        cp_async_commit();
    };

    if (ntiles > 0) load_tile(0, 0);
    __syncthreads();

    for (int t = 0; t < ntiles; ++t) {
        const int buf = t & 1;
        if (t + 1 < ntiles) {
            load_tile(t + 1, buf ^ 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const int t0 = start + t * T;
        const int nk = min(T, end - t0);
        const float *Kt = Ks + (size_t)buf * T * HD;
        const float *Vt = Vs + (size_t)buf * T * HD;

        // scores: warp w takes keys w, w+4, ...; lanes split the head dimension
        for (int j = warp; j < nk; j += kAttnThreads / 32) {
            float kv[HD / 32];
#pragma unroll
            for (int d = 0; d < HD / 32; ++d) kv[d] = Kt[j * HD + d * 32 + lane];
            for (int h = 0; h < G; ++h) {
                float s = 0.f;
#pragma unroll
                for (int d = 0; d < HD / 32; ++d) s = fmaf(qs[h * HD + d * 32 + lane], kv[d], s);
                s = warp_sum(s);
                if (lane == 0) ps[h * T + j] = s * scale;
            }
        }
        __syncthreads();
        // online softmax update, one warp per head
        for (int h = warp; h < G; h += kAttnThreads / 32) {
            float mx = -FLT_MAX;
            for (int j = lane; j < nk; j += 32) mx = fmaxf(mx, ps[h * T + j]);
            mx = warp_max(mx);
            const float m_new = fmaxf(m_run[h], mx);
            float sum = 0.f;
            for (int j = lane; j < nk; j += 32) {
                float e = expf(ps[h * T + j] - m_new);
                ps[h * T + j] = e;
                sum += e;
            }
            sum = warp_sum(sum);
            if (lane == 0) {
                const float c = expf(m_run[h] - m_new);
                corr[h] = c;
                l_run[h] = l_run[h] * c + sum;
                m_run[h] = m_new;
            }
        }
        __syncthreads();
        // o[h][:] = o[h][:] * corr[h] + sum_j p[h][j] V[j][:]
#pragma unroll
        for (int i = 0; i < kSlots; ++i) {
            const int slot = tid + i * kAttnThreads;
            if (slot < G * V4) {
                const int h = slot / V4, c4 = slot % V4;
                const float c = corr[h];
                float4 a = acc[i];
                a.x *= c; a.y *= c; a.z *= c; a.w *= c;
                for (int j = 0; j < nk; ++j) {
                    const float pj = ps[h * T + j];
                    const float4 v = *reinterpret_cast<const float4 *>(Vt + j * HD + c4 * 4);
                    a.x = fmaf(pj, v.x, a.x); a.y = fmaf(pj, v.y, a.y);
                    a.z = fmaf(pj, v.z, a.z); a.w = fmaf(pj, v.w, a.w);
                }
                acc[i] = a;
            }
        }
        __syncthreads();
    }

    // write this slice's unnormalised output and its (max, sum)
#pragma unroll
    for (int i = 0; i < kSlots; ++i) {
        const int slot = tid + i * kAttnThreads;
        if (slot < G * V4) {
            const int h = slot / V4, c4 = slot % V4;
            *reinterpret_cast<float4 *>(part + ((size_t)h * p.splits + split) * (HD + 4) + c4 * 4) = acc[i];
        }
    }
    if (tid < G) {
        float *pp = part + ((size_t)tid * p.splits + split) * (HD + 4);
        pp[HD] = ntiles > 0 ? m_run[tid] : -FLT_MAX;  // record: o[HD], m, l, pad (16-byte aligned)
        pp[HD + 1] = ntiles > 0 ? l_run[tid] : 0.f;
    }
}

// merge the slices of one (row, head): weights exp(m_s - M), normalised by the total sum
template <int HD>
__global__ void k_attn_combine(const AttnParams p) {
    const int h = blockIdx.x, row = blockIdx.y;
    const float *part = p.part + ((size_t)row * p.n_head + h) * p.splits * (HD + 4);
    __shared__ float w_s[256];
    __shared__ float inv_l;
    float M = -FLT_MAX;
    for (int s = 0; s < p.splits; ++s) M = fmaxf(M, part[(size_t)s * (HD + 4) + HD]);
    if (threadIdx.x == 0) {
        float L = 0.f;
        for (int s = 0; s < p.splits; ++s) {
            const float l = part[(size_t)s * (HD + 4) + HD + 1];
            const float w = l > 0.f ? expf(part[(size_t)s * (HD + 4) + HD] - M) : 0.f;
            if (s < 256) w_s[s] = w;
            L += w * l;
        }
        inv_l = 1.f / L;
    }
    __syncthreads();
    for (int d = threadIdx.x; d < HD; d += blockDim.x) {
        float o = 0.f;
        for (int s = 0; s < p.splits; ++s) {
            const float w = s < 256 ? w_s[s] : 0.f;
            if (w != 0.f) o = fmaf(w, part[(size_t)s * (HD + 4) + d], o);
        }
        p.out[(size_t)row * p.ldo + (size_t)h * HD + d] = o * inv_l;
    }
}

template <int HD> void launch_hd(const AttnParams &p, cudaStream_t s) {
    constexpr int T = Tile<HD>::T;
    const size_t smem = (size_t)(4 * T * HD + kMaxG * HD + kMaxG * T) * sizeof(float);
    static bool attr = false;
    if (!attr) {
        cudaFuncSetAttribute(k_attn_split<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        attr = true;
    }
    dim3 grid(p.n_kv, p.splits, p.rows);
    k_attn_split<HD><<<grid, kAttnThreads, smem, s>>>(p);
    k_attn_combine<HD><<<dim3(p.n_head, p.rows), HD < 128 ? HD : 128, 0, s>>>(p);
}

}  // namespace

void launch_attention(const AttnParams &p, cudaStream_t s) {
    switch (p.hd) {
    case 64: return launch_hd<64>(p, s);
    case 128: return launch_hd<128>(p, s);
    case 256: return launch_hd<256>(p, s);
    }
}

}  // namespace syn
