// k_attn.cu -- the standalone split-K decode attention kernel, fed by bulk asynchronous copies: the
// attention operation of "Local inference and architectures" (section "The operations") over the
// KV cache of "Execution contract" (section "Memory lifecycle / KV cache").
//
// One CTA per work item (KV head g, key slice `split`, query row): the keys of a slice are
// contiguous rows of the layer's cache ([n_kv][max_ctx][hd]), so a producer warp streams them with
// cp.async.bulk -- TK keys of K and the same TK keys of V per stage -- into a 3-stage shared-memory
// ring, each stage completing on an mbarrier. Eight consumer warps take KB keys each per stage
// (lane l holds elements l*EL .. l*EL+EL-1 of every row it uses, read conflict-free from shared
// memory), run the same score / online-softmax / output steps as the per-warp streaming form
// (attn_dev.cuh), and release the stage. HBM traffic no longer waits on the consumers: up to three
// stages (192 KB) per SM are in flight.
//
// Keys before the step's first new position were written by earlier steps, so the producer copies
// them before it waits for the previous kernel (programmatic dependent launch); only the stage that
// holds this step's new keys waits. This is sound because the kernel before this one (the per-head
// transforms and KV append, k_heads) releases its dependents only after its own wait: when this
// kernel starts, every earlier kernel -- the previous step's argmax, which advances the position in
// the device state, included -- has completed. Every wait is bounded and reports ERR_ATTN.
//
// In decode with the per-head transforms folded in (fuse_heads; a decode graph replays within one
// step, after the previous step's graph has completed), there is no k_heads before this kernel:
// every CTA transforms its group's query heads in registers (bias, norm_heads, rope), the rings
// stream only keys of earlier steps (no wait at all), and warp 0 of the CTA whose key slice holds
// the new position transforms that position's key, appends key and value to the cache for later
// steps and takes them into its softmax from registers. The transforms' constants (biases,
// head-norm weights, the position's rope factors) are loaded before the wait.
#include "async_dev.cuh"
#include "attn_dev.cuh"
#include "misc_dev.cuh"

namespace syn {

namespace {

constexpr int kRingStages = 3;
constexpr int kRingThreads = kAttnThreads + 32;   // 8 consumer warps + 1 producer warp

// KV: the cache element type (float, or __half for the f16 cache)
template <int HD, int GP, class KV> struct Ring {
    static constexpr int EL = AttnShape<HD, GP>::EL, KB = AttnShape<HD, GP>::KB;
    static constexpr int TK = kAttnWarps * KB;          // keys per stage
    static constexpr int STAGE = 2 * TK * HD;           // elements per stage: K rows, then V rows
    static constexpr size_t SMEM = (size_t)kRingStages * STAGE * sizeof(KV) > attn_smem_bytes<HD, GP>()
                                       ? (size_t)kRingStages * STAGE * sizeof(KV)
                                       : attn_smem_bytes<HD, GP>();   // the merge scratch reuses the ring
};

template <int HD, int GP, class KV>
__global__ void __launch_bounds__(kRingThreads, 1) k_attn(const AttnParams p) {
    using R = Ring<HD, GP, KV>;
    constexpr int EL = R::EL, KB = R::KB, TK = R::TK;
    extern __shared__ __align__(128) float smem_f[];
    KV *ring = reinterpret_cast<KV *>(smem_f);
    __shared__ __align__(8) uint64_t full[kRingStages], empty[kRingStages];
    const int g = blockIdx.x, split = blockIdx.y, row = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kRingStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kAttnWarps);
        }
        mbar_init_fence();
    }
    __syncthreads();
    pdl_launch_dependents();
    int pos, start, end, S;
    attn_range<TK>(p, split, row, pos, start, end, S);
    if (split >= S) return;   // no keys for this item at this step (every thread leaves together)
    // with the per-head transforms folded in (decode: one row), this CTA appends the new position's
    // K/V if its key slice holds that position, and the ring carries only the older keys
    const bool appends = p.fuse_heads && start <= pos && pos < end;
    const int ring_end = p.fuse_heads ? min(end, pos) : end;
    const int nst = ring_end > start ? (ring_end - start + TK - 1) / TK : 0;
    const unsigned spin = p.spin >= 0 ? (unsigned)p.spin : kAsyncSpin;

    if (warp == kAttnWarps) {
        // producer
        if (lane == 0) {
            const KV *Kg = static_cast<const KV *>(p.kcache) + (size_t)g * p.max_ctx * HD;
            const KV *Vg = static_cast<const KV *>(p.vcache) + (size_t)g * p.max_ctx * HD;
            const int first_new = p.state->pos;   // keys from here on are written by this step
            bool waited = false;
            int issued = 0;
            for (int i = 0; i < nst; ++i) {
                const int s = i % kRingStages;
                if (i >= kRingStages && !mbar_wait_n(&empty[s], ((i / kRingStages) - 1) & 1, p.err, ERR_ATTN, spin)) break;
                const int t0 = start + i * TK, nk = min(TK, ring_end - t0);
                if (!waited && t0 + nk > first_new) {
                    // the stage holds keys of this step, written by the previous kernel (never the
                    // case with the per-head transforms folded in)
                    pdl_wait();
                    waited = true;
                }
                KV *sk = ring + s * R::STAGE;
                const unsigned bytes = (unsigned)nk * HD * sizeof(KV);
                mbar_expect_tx(&full[s], 2 * bytes);
                bulk_g2s(sk, Kg + (size_t)t0 * HD, bytes, &full[s]);
                bulk_g2s(sk + TK * HD, Vg + (size_t)t0 * HD, bytes, &full[s]);
                issued = i + 1;
            }
            // no copy may land in shared memory after the CTA has left: wait (with the full
            // bound, whatever `spin` was) for the stages still in flight
            for (int i = max(0, issued - kRingStages); i < issued; ++i)
                mbar_wait(&full[i % kRingStages], (i / kRingStages) & 1, p.err, ERR_ATTN);
        }
        return;
    }

    // consumers
    const int G = p.n_head / p.n_kv;
    float q[GP][EL];
    float kv[EL], vv[EL];   // the new position's key and value (appending CTA, warp 0)
    // with the per-head transforms folded in, their constants (biases, norm weights, the position's
    // rope factors) are weights and tables that no kernel of the step writes: loaded before the wait
    float2 rc[EL];
    float bq[GP][EL], wq[EL], bk[EL], wk[EL], bv[EL];
    if (p.fuse_heads) {
        const HeadsParams &h = p.heads;
        if (h.rope_q || h.rope_k) rope_factors<HD>(rc, h.rope_cs, pos, h.rope_adjacent);
#pragma unroll
        for (int e = 0; e < EL; ++e) {
            const int d = lane * EL + e;
#pragma unroll
            for (int hq = 0; hq < GP; ++hq) bq[hq][e] = h.bq && hq < G ? h.bq[(size_t)(g * G + hq) * HD + d] : 0.f;
            wq[e] = h.wq ? h.wq[d] : 0.f;
            bk[e] = h.bk ? h.bk[(size_t)g * HD + d] : 0.f;
            wk[e] = h.wk ? h.wk[d] : 0.f;
            bv[e] = h.bv ? h.bv[(size_t)g * HD + d] : 0.f;
        }
    }
    pdl_wait();   // q (and k, v) come from the previous kernel
    if (p.fuse_heads) {
        const HeadsParams &h = p.heads;
        if (appends && warp == 0) {
            // transform and append this position's key and value of KV head g (for later steps)
#pragma unroll
            for (int e = 0; e < EL; ++e) {
                kv[e] = __ldcg(h.k + (size_t)g * HD + lane * EL + e);
                vv[e] = __ldcg(h.v + (size_t)g * HD + lane * EL + e) + bv[e];
            }
            head_transform_r<HD>(kv, h.bk != nullptr, bk, h.wk != nullptr, wk, h.rope_k, rc, h.rope_adjacent, h.eps);
            KV *kd = static_cast<KV *>(h.kcache) + ((size_t)g * h.max_ctx + pos) * HD + lane * EL;
            KV *vd = static_cast<KV *>(h.vcache) + ((size_t)g * h.max_ctx + pos) * HD + lane * EL;
#pragma unroll
            for (int e = 0; e < EL; ++e) {
                st_kv(kd + e, kv[e]);
                st_kv(vd + e, vv[e]);
            }
            // the softmax takes the values as stored (rounded to f16 with the f16 cache)
            if constexpr (sizeof(KV) == 2) {
#pragma unroll
                for (int e = 0; e < EL; ++e) {
                    kv[e] = __half2float(__float2half_rn(kv[e]));
                    vv[e] = __half2float(__float2half_rn(vv[e]));
                }
            }
        }
#pragma unroll
        for (int hq = 0; hq < GP; ++hq) {
            if (hq < G) {
                const int qh = g * G + hq;
#pragma unroll
                for (int e = 0; e < EL; ++e) q[hq][e] = __ldcg(h.q + (size_t)qh * HD + lane * EL + e);
                head_transform_r<HD>(q[hq], h.bq != nullptr, bq[hq], h.wq != nullptr, wq, h.rope_q, rc, h.rope_adjacent, h.eps);
            } else {
#pragma unroll
                for (int e = 0; e < EL; ++e) q[hq][e] = 0.f;
            }
        }
    } else {
        attn_load_q<HD, GP>(p, g, row, q);
    }
    const float scale = 1.f / sqrtf((float)HD);
    float m_run = -FLT_MAX, l_run = 0.f;
    float o[GP][EL];
#pragma unroll
    for (int h = 0; h < GP; ++h)
#pragma unroll
        for (int e = 0; e < EL; ++e) o[h][e] = 0.f;
    if (appends && warp == 0) {   // the new key, from registers
        float kr[KB][EL], vr[KB][EL];
#pragma unroll
        for (int j = 0; j < KB; ++j)
#pragma unroll
            for (int e = 0; e < EL; ++e) {
                kr[j][e] = j == 0 ? kv[e] : 0.f;
                vr[j][e] = j == 0 ? vv[e] : 0.f;
            }
        attn_step<HD, GP>(q, kr, vr, 1, G, scale, m_run, l_run, o);
    }
    for (int i = 0; i < nst; ++i) {
        const int s = i % kRingStages;
        if (!mbar_wait_n(&full[s], (i / kRingStages) & 1, p.err, ERR_ATTN, spin)) break;
        const int t0 = start + i * TK + warp * KB;
        const int nk = min(KB, ring_end - t0);
        if (nk > 0) {
            const KV *sk = ring + s * R::STAGE + warp * KB * HD + lane * EL;
            const KV *sv = sk + TK * HD;
            float kr[KB][EL], vr[KB][EL];
#pragma unroll
            for (int j = 0; j < KB; ++j) {
                if (j < nk) {
                    lds_row<EL>(kr[j], sk + j * HD);
                    lds_row<EL>(vr[j], sv + j * HD);
                } else {
#pragma unroll
                    for (int e = 0; e < EL; ++e) { kr[j][e] = 0.f; vr[j][e] = 0.f; }
                }
            }
            attn_step<HD, GP>(q, kr, vr, nk, G, scale, m_run, l_run, o);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
    // every stage has been consumed (or the wait gave up): the ring is free for the merge
    bar_sync_first(kAttnThreads);
    attn_finish<HD, GP>(p, S, g, split, row, smem_f, m_run, l_run, o, [] { bar_sync_first(kAttnThreads); });
}

template <int HD, int GP, class KV> void launch_kv(const AttnParams &p, cudaStream_t s, bool pdl) {
    constexpr size_t smem = Ring<HD, GP, KV>::SMEM;
    // a failure here makes the launch below fail, and that error reaches the caller
    ensure_dyn_smem(reinterpret_cast<const void *>(k_attn<HD, GP, KV>), (int)smem);
    if (pdl)
        launch_pdl(k_attn<HD, GP, KV>, dim3(p.n_kv, p.splits, p.rows), dim3(kRingThreads), smem, s, p);
    else
        k_attn<HD, GP, KV><<<dim3(p.n_kv, p.splits, p.rows), kRingThreads, smem, s>>>(p);
}

template <int HD, int GP> void launch_t(const AttnParams &p, cudaStream_t s, bool pdl) {
    if (p.kv_f16) launch_kv<HD, GP, __half>(p, s, pdl);
    else launch_kv<HD, GP, float>(p, s, pdl);
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
