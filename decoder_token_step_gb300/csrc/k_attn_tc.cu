// k_attn_tc.cu -- bulk-prefill attention on the 5th-generation tensor cores (tcgen05, TMEM, TMA).
//
// `attention(q, k, v)` of "Local inference and architectures" (section "The format": causal
// attention over the cache, GQA, sliding windows where the architecture has them) for the n rows of
// a bulk prefill ("Execution contract", section "Prefill"): row i sits at position pos + i and
// attends to the cached keys t <= pos + i (t > pos + i - window on windowed layers). Per query head
// this is S = Q K^T / sqrt(hd), a causal softmax over each row, and O = P V -- two dense products
// that go to the tensor cores, with the softmax between them on the CUDA cores, key tile by key
// tile (online softmax: a running row maximum and row sum rescale the partial output).
//
// The decoder computes in f32, so every product uses the same f32-grade split as the bulk GEMM
// (k_gemm_tc.cu): an operand vector scaled by a power of two s (its largest magnitude just under
// 2^14) is split into f16 halves, v s = vh + vl, and a b ~= (ah bh + ah bl + al bh) / (sa sb) keeps
// 22 significant bits of each operand. Scales: per query row of Q (undone on that row of S), per key
// row of K (undone on that column of S), per 64-key tile of V (undone when the tile's partial output
// is added), none for P (its entries lie in [0, 2^8]).
//
// Three kernels per attention node:
//   k_attn_split_q   q rows (f32) -> Qh, Ql [n_head][Rp][hd] (Rp = n rounded up to 128) + 1/s per row
//   k_attn_split_kv  cache keys 0 .. pos + n - 1 (f32 or f16) -> Kh, Kl [n_kv][Lp][hd] + 1/s per key,
//                    and V transposed, Vh, Vl [n_kv][hd][Lp] (keys contiguous, the K-major layout the
//                    P V product needs) + 1/s per 64-key tile; the rest of the last tile is zero
//   k_attn_tc        one CTA per (query head, 128-row query block), the blocks with the most key
//                    tiles first:
//       warp 0       TMA producer: Q hi/lo once, then per 64-key tile K hi/lo (with the tile's
//                    scales) and V^T hi/lo into two 2-slot rings (128-byte swizzle, mbarrier
//                    completion): a K slot is refilled once S of its tile is done, a V slot once
//                    P V is, so the next tiles load while the tensor core works;
//       warp 1       allocates 512 TMEM columns (two 128 x 128 f32 score buffers, one 128 x 2 hd
//                    output buffer); one thread issues S(t) = Q K(t)^T (2 MMAs per 16-wide k step:
//                    Qh [Kh | Kl]^T and Ql Kh^T), then O(t-1) = P(t-1) V(t-1) (Ph [Vh | Vl]^T and
//                    Pl Vh^T) once the softmax has written P(t-1) -- so the scores of tile t are
//                    computed while the softmax of tile t-1 runs;
//       warps 2..9   softmax, two warps per 32 query rows (TMEM lanes = rows): both read S(t) and
//                    take the row's maximum; each then handles half of the row -- exponentials (in
//                    base 2, against a reference maximum that moves only when the row maximum
//                    grows by more than a factor 2^8; the mask only on tiles that cross an edge)
//                    and partial sum of 32 keys, its half of the previous tile's O (read from TMEM,
//                    times its V scale) added into f32 registers, rescaled when the reference
//                    moved, its half of P(t) written as f16 hi/lo into shared memory in the
//                    swizzled K-major layout of an MMA A operand; at the end O / sum is stored.
// The output of each tile is accumulated by the tensor core over only 64 keys and summed in f32
// registers, as in the GEMM (its accumulation is not rounded to nearest).
//
// Every wait is bounded: a wait that runs out sets ERR_ATTN in the device state and the CTA winds
// down (it still waits, bounded, for its copies and MMAs in flight before freeing TMEM).
#include <algorithm>
#include <type_traits>

#include "tc_dev.cuh"

namespace syn {

namespace {

template <int HD> struct Atc {
    static constexpr int BQ = 128;                   // query rows per CTA (MMA M)
    static constexpr int BK = 64;                    // keys per tile (N of S, K of P V)
    static constexpr int NB = HD / 64;               // 64-wide boxes along the head dimension
    static constexpr int Q_BOX = BQ * 128;           // bytes of one 128-row x 64-column f16 box
    static constexpr int K_BOX = BK * 128;
    static constexpr int Q_PLANE = NB * Q_BOX;       // one of Qh, Ql
    static constexpr int K_PLANE = NB * K_BOX;       // one of Kh, Kl (one tile)
    static constexpr int V_PLANE = HD * 128;         // one of Vh, Vl: hd rows x 64 keys
    static constexpr int P_PLANE = BQ * 128;         // one of Ph, Pl: 128 rows x 64 keys
    static constexpr int K_STAGE = 2 * K_PLANE;      // Kh, Kl of one tile
    static constexpr int V_STAGE = 2 * V_PLANE;      // Vh, Vl of one tile
    static constexpr int STAGES = 2;                 // slots of the K ring and of the V ring
    static constexpr int SCALES = BK * 4 + 16;       // 1/s of the tile's keys, then the V tile's 1/s
    static constexpr int SC_SLOTS = 4;
    static constexpr int SMEM =
        1024 + 2 * Q_PLANE + STAGES * (K_STAGE + V_STAGE) + 2 * P_PLANE + SC_SLOTS * SCALES;
    static constexpr int THREADS = 64 + 256;          // producer, MMA, 8 softmax warps
    // TMEM: two S buffers of 128 columns (Qh Kh^T + Ql Kh^T in the first 64, Qh Kl^T in the other
    // 64), then O: Ph Vh^T + Pl Vh^T in hd columns, Ph Vl^T in the next hd
    static constexpr int S_COLS = 2 * BK;
    static constexpr int O_COL = 2 * S_COLS;
    static constexpr int TMEM_COLS = 512;
    static_assert(HD == 64 || HD == 128, "head size");
};

constexpr int kSplitThreads = 256;

// q [rows][n_head * hd] (row stride ldq) -> scaled hi/lo planes [n_head][Rp][hd] and 1/scale per
// (head, row); rows rows .. Rp-1 are zero. One warp per (head, row).
template <int HD>
__global__ void __launch_bounds__(kSplitThreads) k_attn_split_q(const float *q, int64_t ldq, int rows, int Rp, int n_head,
                                                                 __half *qh, __half *ql, float *inv_s) {
    constexpr int EL = HD / 32;
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int item = blockIdx.x * (kSplitThreads / 32) + (threadIdx.x >> 5);
    if (item >= n_head * Rp) return;
    const int h = item / Rp, r = item % Rp;
    float v[EL];
    float amax = 0.f;
#pragma unroll
    for (int e = 0; e < EL; ++e) {
        v[e] = r < rows ? q[(size_t)r * ldq + (size_t)h * HD + lane * EL + e] : 0.f;
        amax = fmaxf(amax, fabsf(v[e]));
    }
    const float sc = row_scale(warp_max(amax));
    __half hi[EL], lo[EL];
#pragma unroll
    for (int e = 0; e < EL; ++e) split2(v[e] * sc, hi[e], lo[e]);
    const size_t off = (size_t)item * HD + lane * EL;
    if constexpr (EL == 4) {
        *reinterpret_cast<uint2 *>(qh + off) = *reinterpret_cast<const uint2 *>(hi);
        *reinterpret_cast<uint2 *>(ql + off) = *reinterpret_cast<const uint2 *>(lo);
    } else {
        *reinterpret_cast<uint32_t *>(qh + off) = *reinterpret_cast<const uint32_t *>(hi);
        *reinterpret_cast<uint32_t *>(ql + off) = *reinterpret_cast<const uint32_t *>(lo);
    }
    if (lane == 0) inv_s[item] = 1.f / sc;
}

SYN_DEV float ld_kv(const float *p) { return __ldcg(p); }
SYN_DEV float ld_kv(const __half *p) { return __half2float(*p); }

// One CTA per (64-key tile, KV head) of keys 0 .. pos + rows - 1 of one layer's cache
// ([n_kv][max_ctx][hd]); tiles past the last key return at once. Keys past the last one in the
// last tile are written as zero (scale 1), so the attention reads only finite values.
template <int HD, class KV>
__global__ void __launch_bounds__(kSplitThreads) k_attn_split_kv(const KV *kc, const KV *vc, int max_ctx, int Lp, int rows,
                                                                  const DevState *state, __half *kh, __half *kl,
                                                                  float *inv_sk, __half *vh, __half *vl, float *inv_sv) {
    constexpr int EL = HD / 32, BK = 64, NW = kSplitThreads / 32;
    __shared__ float vs[BK][HD + 1];
    __shared__ float red[NW];
    pdl_wait();
    const int kend = state->pos + rows;
    const int t = blockIdx.x, g = blockIdx.y, t0 = t * BK;
    if (t0 >= kend) return;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const KV *kg = kc + (size_t)g * max_ctx * HD;
    const KV *vg = vc + (size_t)g * max_ctx * HD;

    // keys: one warp per key row, per-row scale
    for (int j = warp; j < BK; j += NW) {
        const int key = t0 + j;
        float v[EL];
        float amax = 0.f;
#pragma unroll
        for (int e = 0; e < EL; ++e) {
            v[e] = key < kend ? ld_kv(kg + (size_t)key * HD + lane * EL + e) : 0.f;
            amax = fmaxf(amax, fabsf(v[e]));
        }
        const float sc = row_scale(warp_max(amax));
        __half hi[EL], lo[EL];
#pragma unroll
        for (int e = 0; e < EL; ++e) split2(v[e] * sc, hi[e], lo[e]);
        const size_t off = ((size_t)g * Lp + key) * HD + lane * EL;
        if constexpr (EL == 4) {
            *reinterpret_cast<uint2 *>(kh + off) = *reinterpret_cast<const uint2 *>(hi);
            *reinterpret_cast<uint2 *>(kl + off) = *reinterpret_cast<const uint2 *>(lo);
        } else {
            *reinterpret_cast<uint32_t *>(kh + off) = *reinterpret_cast<const uint32_t *>(hi);
            *reinterpret_cast<uint32_t *>(kl + off) = *reinterpret_cast<const uint32_t *>(lo);
        }
        if (lane == 0) inv_sk[(size_t)g * Lp + key] = 1.f / sc;
    }

    // values: the tile through shared memory, one scale for the tile, written transposed
    float amax = 0.f;
    for (int i = threadIdx.x; i < BK * HD; i += kSplitThreads) {
        const int j = i / HD, d = i % HD, key = t0 + j;
        const float v = key < kend ? ld_kv(vg + (size_t)key * HD + d) : 0.f;
        vs[j][d] = v;
        amax = fmaxf(amax, fabsf(v));
    }
    amax = warp_max(amax);
    if (lane == 0) red[warp] = amax;
    __syncthreads();
    amax = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) amax = fmaxf(amax, red[w]);
    const float sc = row_scale(amax);
    // item = (d, 8-key chunk): 8 consecutive keys of row d of V^T, one 16-byte store per plane
    for (int i = threadIdx.x; i < HD * (BK / 8); i += kSplitThreads) {
        const int d = i / (BK / 8), c = i % (BK / 8);
        __half hi[8], lo[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) split2(vs[c * 8 + e][d] * sc, hi[e], lo[e]);
        const size_t off = ((size_t)g * HD + d) * Lp + t0 + c * 8;
        *reinterpret_cast<uint4 *>(vh + off) = *reinterpret_cast<const uint4 *>(hi);
        *reinterpret_cast<uint4 *>(vl + off) = *reinterpret_cast<const uint4 *>(lo);
    }
    if (threadIdx.x < 4) inv_sv[((size_t)g * (Lp / BK) + t) * 4 + threadIdx.x] = 1.f / sc;
}

struct AtcArgs {
    float *out;
    int64_t ldo;
    const float *inv_sq;   // [n_head][Rp]
    const float *inv_sk;   // [n_kv][Lp]
    const float *inv_sv;   // [n_kv][Lp / 64][4]
    const DevState *state;
    int *err;
    int rows, Rp, Lp, n_head, n_kv, window;
};

// 8 f32 values -> 8 f16 hi halves and 8 f16 lo halves (two 16-byte chunks), two values per
// conversion; the same halves as split2
SYN_DEV void split8(const float *p, uint4 &h, uint4 &l) {
    uint32_t hh[4], ll[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const __half2 hv = __floats2half2_rn(p[2 * e], p[2 * e + 1]);
        const float2 back = __half22float2(hv);
        const __half2 lv = __floats2half2_rn(p[2 * e] - back.x, p[2 * e + 1] - back.y);
        hh[e] = *reinterpret_cast<const uint32_t *>(&hv);
        ll[e] = *reinterpret_cast<const uint32_t *>(&lv);
    }
    h = make_uint4(hh[0], hh[1], hh[2], hh[3]);
    l = make_uint4(ll[0], ll[1], ll[2], ll[3]);
}

// 2^x with the hardware approximation (relative error of order 2^-22; -inf gives 0)
SYN_DEV float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

constexpr float kLog2E = 1.4426950408889634f;   // log2(e): exp(x) = 2^(x log2 e)

// a bounded wait taken by a whole warp, with one answer for all its lanes (so that no lane leaves a
// loop that the others stay in)
SYN_DEV bool warp_wait(uint64_t *bar, unsigned parity, int *err) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, err, ERR_ATTN));
}

template <int HD>
__global__ void __launch_bounds__(Atc<HD>::THREADS, 1)
    k_attn_tc(const __grid_constant__ CUtensorMap mQh, const __grid_constant__ CUtensorMap mQl,
              const __grid_constant__ CUtensorMap mKh, const __grid_constant__ CUtensorMap mKl,
              const __grid_constant__ CUtensorMap mVh, const __grid_constant__ CUtensorMap mVl, const AtcArgs a) {
    using A = Atc<HD>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sQh = base, *sQl = base + A::Q_PLANE;
    uint8_t *kring = base + 2 * A::Q_PLANE, *vring = kring + A::STAGES * A::K_STAGE;
    uint8_t *sPh = vring + A::STAGES * A::V_STAGE, *sPl = sPh + A::P_PLANE;
    uint8_t *scales = sPl + A::P_PLANE;
    __shared__ __align__(8) uint64_t q_full, k_full[2], k_empty[2], v_full[2], v_empty[2], sc_full[A::SC_SLOTS],
        s_full[2], s_empty[2], p_full, o_full, done, l_ready;
    __shared__ uint32_t tmem_base;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // work item: the query blocks with the most key tiles first; heads of one KV head side by side
    const int nqb = a.Rp / A::BQ;
    const int h = blockIdx.x % a.n_head, qb = nqb - 1 - (int)(blockIdx.x / a.n_head);
    const int g = h / (a.n_head / a.n_kv);
    const int i0 = qb * A::BQ;

    if (threadIdx.x == 0) {
        mbar_init(&q_full, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 1);
            mbar_init(&v_full[s], 1);
            mbar_init(&v_empty[s], 1);
            mbar_init(&s_full[s], 1);
            mbar_init(&s_empty[s], 8);   // one arrival per softmax warp
        }
        for (int s = 0; s < A::SC_SLOTS; ++s) mbar_init(&sc_full[s], 1);
        mbar_init(&p_full, 8);
        mbar_init(&l_ready, 256);   // every softmax thread
        mbar_init(&o_full, 1);
        mbar_init(&done, 1);
        mbar_init_fence();
    }
    if (warp == 1) tmem_alloc(&tmem_base, A::TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;
    pdl_wait();   // the split planes come from the kernels just before

    // key tiles of this block: from the first key the block's first row may see to the last row's own
    const int pos0 = a.state->pos;
    const int q_lo = pos0 + i0, q_hi = pos0 + min(i0 + A::BQ, a.rows) - 1;
    const int key_lo = a.window > 0 ? max(0, q_lo - a.window + 1) : 0;
    const int t_first = key_lo / A::BK, nt = q_hi / A::BK - t_first + 1;

    if (warp == 0) {
        if (lane == 0) {
            // K(t) may load once S(t-2) is done with its slot, V(t) once P V(t-2) is; the tensor core
            // finishes S(t-1) before P V(t-2), so K runs one tile ahead of V. The tile's scales go
            // to a 4-slot ring of their own (the softmax reads them until it has written P(t)).
            bool ok = true;
            int k_issued = 0, v_issued = 0;
            mbar_expect_tx(&q_full, 2 * A::Q_PLANE);
            for (int b = 0; b < A::NB; ++b) {
                tma_load_2d(sQh + b * A::Q_BOX, &mQh, b * 64, h * a.Rp + i0, &q_full);
                tma_load_2d(sQl + b * A::Q_BOX, &mQl, b * 64, h * a.Rp + i0, &q_full);
            }
            for (int step = 0; step <= nt && ok; ++step) {
                if (step < nt) {
                    const int it = step, s = it & 1, t = t_first + it;
                    if (it >= 2 && !(ok = mbar_wait(&k_empty[s], ((it >> 1) - 1) & 1, a.err, ERR_ATTN))) break;
                    uint8_t *ks = kring + s * A::K_STAGE;
                    mbar_expect_tx(&k_full[s], A::K_STAGE);
                    // per 64-wide head block b: the Kh box, then the Kl box -- one 128-row operand
                    for (int b = 0; b < A::NB; ++b) {
                        tma_load_2d(ks + 2 * b * A::K_BOX, &mKh, b * 64, g * a.Lp + t * A::BK, &k_full[s]);
                        tma_load_2d(ks + (2 * b + 1) * A::K_BOX, &mKl, b * 64, g * a.Lp + t * A::BK, &k_full[s]);
                    }
                    uint8_t *sc = scales + (it % A::SC_SLOTS) * A::SCALES;
                    uint64_t *scb = &sc_full[it % A::SC_SLOTS];
                    mbar_expect_tx(scb, A::SCALES);
                    bulk_g2s(sc, a.inv_sk + (size_t)g * a.Lp + t * A::BK, A::BK * 4, scb);
                    bulk_g2s(sc + A::BK * 4, a.inv_sv + ((size_t)g * (a.Lp / A::BK) + t) * 4, 16, scb);
                    k_issued = it + 1;
                }
                if (step >= 1) {
                    const int it = step - 1, s = it & 1, t = t_first + it;
                    if (it >= 2 && !(ok = mbar_wait(&v_empty[s], ((it >> 1) - 1) & 1, a.err, ERR_ATTN))) break;
                    uint8_t *vs = vring + s * A::V_STAGE;
                    mbar_expect_tx(&v_full[s], A::V_STAGE);
                    tma_load_2d(vs, &mVh, t * A::BK, g * HD, &v_full[s]);
                    tma_load_2d(vs + A::V_PLANE, &mVl, t * A::BK, g * HD, &v_full[s]);
                    v_issued = it + 1;
                }
            }
            // nothing may land in shared memory after the CTA has gone: wait for the copies in flight
            mbar_wait(&q_full, 0, a.err, ERR_ATTN);
            for (int it = max(0, k_issued - 2); it < k_issued; ++it)
                mbar_wait(&k_full[it & 1], (it >> 1) & 1, a.err, ERR_ATTN);
            for (int it = max(0, k_issued - A::SC_SLOTS); it < k_issued; ++it)
                mbar_wait(&sc_full[it % A::SC_SLOTS], (it / A::SC_SLOTS) & 1, a.err, ERR_ATTN);
            for (int it = max(0, v_issued - 2); it < v_issued; ++it)
                mbar_wait(&v_full[it & 1], (it >> 1) & 1, a.err, ERR_ATTN);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // The three products of a split share operands: Kh and Kl (Vh and Vl) sit one after the
            // other, so Qh [Kh | Kl]^T (Ph [Vh | Vl]^T) is one MMA twice as wide, and only Ql Kh^T (Pl
            // Vh^T) is a second one -- fewer, wider MMAs, whose issue is what bounds this thread.
            constexpr uint32_t idS2 = tc_idesc_f16(A::BQ, 2 * A::BK), idS1 = tc_idesc_f16(A::BQ, A::BK);
            constexpr uint32_t idO2 = tc_idesc_f16(A::BQ, 2 * HD), idO1 = tc_idesc_f16(A::BQ, HD);
            const uint64_t dqh = desc_sw128(saddr(sQh)), dql = desc_sw128(saddr(sQl));
            const uint64_t dph = desc_sw128(saddr(sPh)), dpl = desc_sw128(saddr(sPl));
            // O(t) = P(t) V(t): 4 k steps of 16 keys into a fresh accumulator (the softmax warps
            // drained O(t-1) from it before they released P(t))
            auto issue_pv = [&](int it) {
                const uint64_t dv = desc_sw128(saddr(vring + (it & 1) * A::V_STAGE));
                const uint32_t d = tmem + A::O_COL;
#pragma unroll
                for (int k = 0; k < A::BK / 16; ++k) {
                    const uint32_t off = desc_off(k * 32);
                    mma_f16(d, dph + off, dv + off, idO2, k != 0);
                    mma_f16(d, dpl + off, dv + off, idO1, 1);
                }
            };
            bool ok = mbar_wait(&q_full, 0, a.err, ERR_ATTN);
            for (int it = 0; it < nt && ok; ++it) {
                const int s = it & 1, b = it & 1;
                // K(it) landed; for it >= 2 the softmax warps also read S(it-2) out of buffer b
                ok = it >= 2 ? mbar_wait2(&k_full[s], (it >> 1) & 1, &s_empty[b], ((it >> 1) - 1) & 1, a.err, ERR_ATTN)
                             : mbar_wait(&k_full[s], (it >> 1) & 1, a.err, ERR_ATTN);
                if (!ok) break;
                tc_fence_after();
                const uint64_t dk = desc_sw128(saddr(kring + s * A::K_STAGE));
                const uint32_t d = tmem + (uint32_t)(b * A::S_COLS);
#pragma unroll
                for (int k = 0; k < HD / 16; ++k) {
                    const uint32_t qo = desc_off((k >> 2) * A::Q_BOX + (k & 3) * 32);
                    const uint32_t ko = desc_off((k >> 2) * 2 * A::K_BOX + (k & 3) * 32);
                    mma_f16(d, dqh + qo, dk + ko, idS2, k != 0);
                    mma_f16(d, dql + qo, dk + ko, idS1, 1);
                }
                mma_commit(&s_full[b]);
                mma_commit(&k_empty[s]);   // the K slot is free once S(it) is done
                if (it >= 1) {
                    // V(it-1) landed (long since), P(it-1) written (and O(it-2) drained) by the softmax
                    // warps
                    if (!(ok = mbar_wait2(&v_full[(it - 1) & 1], ((it - 1) >> 1) & 1, &p_full, (it - 1) & 1, a.err,
                                            ERR_ATTN)))
                        break;
                    tc_fence_after();
                    issue_pv(it - 1);
                    mma_commit(&o_full);
                    mma_commit(&v_empty[(it - 1) & 1]);
                }
            }
            if (ok && nt >= 1 && mbar_wait(&p_full, (nt - 1) & 1, a.err, ERR_ATTN) &&
                mbar_wait(&v_full[(nt - 1) & 1], ((nt - 1) >> 1) & 1, a.err, ERR_ATTN)) {
                tc_fence_after();
                issue_pv(nt - 1);
                mma_commit(&o_full);
            }
            mma_commit(&done);   // arrives when every MMA issued above has completed
        }
    } else {
        // softmax: warp w reads TMEM lanes 32 (w % 4) .. + 31, i.e. query rows r of the block, and
        // owns half hf = (w - 2) / 4 of the work on them: the exponentials and P entries of score
        // columns hf * 32 .. + 31 of each key tile, and output columns hf * hd/2 .. + hd/2 - 1. Both
        // warps of a row read all 64 scores and take the same maximum (same values; the maximum does
        // not depend on the order); their partial row sums are added at the end.
        //
        // Scores are kept as u = S / s_k (the query scale and 1/sqrt(hd) folded into c, together with
        // log2 e), so exp(score - m) = 2^(u c - m c): one FMA and one ex2 per entry. The reference
        // maximum m moves only when a tile raises the row maximum by more than 2^kTau in the
        // exponential's terms (entries of P then stay below 2^kTau, far inside the f16 range of its
        // halves); any reference gives the same softmax once O is divided by the row sum, and the
        // warps' registers need no rescaling while it stays put.
        constexpr int SC = A::BK / 2, OC = HD / 2;
        constexpr float kTau = 8.f;
        const int qw = warp & 3, hf = (warp - 2) >> 2, r = qw * 32 + lane, i = i0 + r;
        const int qpos = pos0 + i;
        const int wlo = a.window > 0 ? qpos - a.window + 1 : 0;   // first allowed key
        // a tile needs no mask for any row of this warp when its last key is at or before the warp's
        // first query position and its first key at or after the latest window start of the warp
        const int qpos_w = pos0 + i0 + qw * 32;
        const int wlo_w = a.window > 0 ? qpos_w + 31 - a.window + 1 : 0;
        const uint32_t lane_base = tmem + ((uint32_t)(qw * 32) << 16);
        const float c = a.inv_sq[(size_t)h * a.Rp + i] * (1.f / sqrtf((float)HD)) * kLog2E;
        float o[OC];
#pragma unroll
        for (int d = 0; d < OC; ++d) o[d] = 0.f;
        float m_ref = -1e30f, nmc = 1e30f * c, l_run = 0.f, isv_prev = 0.f;
        bool ok = true;
        // this warp's columns of O(t-1) (relative to the previous reference; the sum of its two
        // column groups) added into o, then o rescaled by alpha when some row of the warp moved its
        // reference
        auto drain = [&](float isv, float alpha, bool rescale) {
#pragma unroll
            for (int c0 = 0; c0 < OC; c0 += 16) {   // 16 columns of each group at a time (P is live)
                uint32_t ra[16], rb[16];
                tmem_ld16_issue(lane_base + A::O_COL + (uint32_t)(hf * OC + c0), ra);
                tmem_ld16_issue(lane_base + A::O_COL + (uint32_t)(HD + hf * OC + c0), rb);
                tmem_ld_wait();
                if (rescale) {
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        o[c0 + j] = fmaf(__uint_as_float(ra[j]) + __uint_as_float(rb[j]), isv, o[c0 + j]) * alpha;
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        o[c0 + j] = fmaf(__uint_as_float(ra[j]) + __uint_as_float(rb[j]), isv, o[c0 + j]);
                }
            }
        };
        for (int it = 0; it < nt; ++it) {
            const int b = it & 1, t = t_first + it, key0 = t * A::BK;
            // the tile's scales were written by a bulk copy: observe their barrier (the slot is loaded
            // again for tile it + 4 only once S(it + 2) is done, which the MMA thread issues after
            // this thread has released P(it)); both tests go out together
            if (!(ok = __all_sync(0xffffffffu, mbar_wait2(&sc_full[it % A::SC_SLOTS], (it / A::SC_SLOTS) & 1,
                                                            &s_full[b], (it >> 1) & 1, a.err, ERR_ATTN))))
                break;
            tc_fence_after();
            const float *sk = reinterpret_cast<const float *>(scales + (it % A::SC_SLOTS) * A::SCALES);
            // u of the other half's 32 keys (only their maximum is kept), then of this warp's own 32;
            // the mask only on tiles that cross a causal or window edge of some row of the warp
            float p[SC];
            float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};   // four independent chains
            auto scan = [&](auto masked) {
                // a score is the sum of its two column groups, times the key's 1/s_k, masked
                auto score = [&](uint32_t x, uint32_t y, float skj, int key) {
                    float v = (__uint_as_float(x) + __uint_as_float(y)) * skj;
                    if constexpr (decltype(masked)::value) v = key <= qpos && key >= wlo ? v : -INFINITY;
                    return v;
                };
                const uint32_t sb = lane_base + (uint32_t)(b * A::S_COLS);
                {   // the other half, 16 columns of each group at a time: only the maximum kept
                    const int cb = (hf ^ 1) * SC;
#pragma unroll
                    for (int q = 0; q < SC; q += 16) {
                        uint32_t ra[16], rb[16];
                        tmem_ld16_issue(sb + cb + q, ra);
                        tmem_ld16_issue(sb + A::BK + cb + q, rb);
                        tmem_ld_wait();
                        const float4 *sk4 = reinterpret_cast<const float4 *>(sk + cb + q);
#pragma unroll
                        for (int j4 = 0; j4 < 4; ++j4) {
                            const float4 s4 = sk4[j4];
                            const float sv[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                const int j = j4 * 4 + e;
                                mx4[e] = fmaxf(mx4[e], score(ra[j], rb[j], sv[e], key0 + cb + q + j));
                            }
                        }
                    }
                }
                // this warp's half, 16 columns of each group at a time, kept in p
                const int cb = hf * SC;
#pragma unroll
                for (int q = 0; q < SC; q += 16) {
                    uint32_t ra[16], rb[16];
                    tmem_ld16_issue(sb + cb + q, ra);
                    tmem_ld16_issue(sb + A::BK + cb + q, rb);
                    tmem_ld_wait();
                    const float4 *sk4 = reinterpret_cast<const float4 *>(sk + cb + q);
#pragma unroll
                    for (int j4 = 0; j4 < 4; ++j4) {
                        const float4 s4 = sk4[j4];
                        const float sv[4] = {s4.x, s4.y, s4.z, s4.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int j = j4 * 4 + e;
                            p[q + j] = score(ra[j], rb[j], sv[e], key0 + cb + q + j);
                            mx4[e] = fmaxf(mx4[e], p[q + j]);
                        }
                    }
                }
            };
            if (key0 + A::BK - 1 <= qpos_w && key0 >= wlo_w)
                scan(std::false_type{});
            else
                scan(std::true_type{});
            const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_empty[b]);
            // move the reference when the tile raised the maximum by more than 2^kTau (a fully
            // masked tile leaves mx = -inf and never moves it)
            const bool move = (mx - m_ref) * c > kTau;
            float alpha = 1.f;
            if (move) {
                alpha = ex2_approx((m_ref - mx) * c);
                m_ref = mx;
                nmc = -mx * c;
            }
            float s0 = 0.f, s1 = 0.f;
#pragma unroll
            for (int j = 0; j < SC; j += 2) {
                p[j] = ex2_approx(fmaf(p[j], c, nmc));   // 2^-inf = 0 for the masked keys
                p[j + 1] = ex2_approx(fmaf(p[j + 1], c, nmc));
                s0 += p[j];
                s1 += p[j + 1];
            }
            l_run = fmaf(l_run, alpha, s0 + s1);
            const float isv = sk[A::BK];
            if (it >= 1) {
                // P V(it-1) is complete: P's buffer is free, O(it-1) can be read
                if (!(ok = warp_wait(&o_full, (it - 1) & 1, a.err))) break;
                tc_fence_after();
                drain(isv_prev, alpha, __any_sync(0xffffffffu, move));
            }
            isv_prev = isv;
            // this warp's half of P(it) as f16 hi/lo, row r of a 128-byte-swizzled K-major tile:
            // 16-byte chunk c of the row goes to chunk c ^ (r mod 8)
#pragma unroll
            for (int cc = 0; cc < SC / 8; ++cc) {
                const int ch = hf * (SC / 8) + cc;
                uint4 hv, lv;
                split8(p + cc * 8, hv, lv);
                const int off = r * 128 + ((ch ^ (r & 7)) << 4);
                *reinterpret_cast<uint4 *>(sPh + off) = hv;
                *reinterpret_cast<uint4 *>(sPl + off) = lv;
            }
            fence_proxy_async_smem();
            tc_fence_before();   // the drain of O(it-1) is ordered before this release
            __syncwarp();
            if (lane == 0) mbar_arrive(&p_full);
        }
        if (ok && nt >= 1 && warp_wait(&o_full, (nt - 1) & 1, a.err)) {
            tc_fence_after();
            drain(isv_prev, 1.f, false);
            // the two partial row sums meet in P's buffer, free now that the last P V is done
            float *lsum = reinterpret_cast<float *>(sPh);
            lsum[hf * A::BQ + r] = l_run;
            mbar_arrive(&l_ready);
            if (mbar_wait(&l_ready, 0, a.err, ERR_ATTN) && i < a.rows) {
                const float inv_l = 1.f / (l_run + lsum[(hf ^ 1) * A::BQ + r]);
                float *dst = a.out + (size_t)i * a.ldo + (size_t)h * HD + hf * OC;
#pragma unroll
                for (int d = 0; d < OC; d += 4)
                    *reinterpret_cast<float4 *>(dst + d) = make_float4(o[d] * inv_l, o[d + 1] * inv_l, o[d + 2] * inv_l, o[d + 3] * inv_l);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        // the columns are freed only after every committed MMA has finished with them
        if (lane == 0) mbar_wait(&done, 0, a.err, ERR_ATTN);
        __syncwarp();
        tc_fence_after();
        tmem_free(tmem, A::TMEM_COLS);
    }
}

int round_up(int v, int m) { return (v + m - 1) / m * m; }

struct Planes {
    __half *qh, *ql, *kh, *kl, *vh, *vl;
    float *inv_sq, *inv_sk, *inv_sv;
};

// q scratch: [Qh][Ql][1/s per (head, row)]; kv scratch: [Kh][Kl][Vh][Vl][1/s per key][1/s per tile x 4]
Planes planes(const AttnParams &p, void *qs, void *kvs) {
    const size_t Rp = round_up(p.rows, 128), Lp = round_up(p.max_ctx, 64);
    Planes P;
    P.qh = static_cast<__half *>(qs);
    P.ql = P.qh + (size_t)p.n_head * Rp * p.hd;
    P.inv_sq = reinterpret_cast<float *>(P.ql + (size_t)p.n_head * Rp * p.hd);
    const size_t kv = (size_t)p.n_kv * Lp * p.hd;
    P.kh = static_cast<__half *>(kvs);
    P.kl = P.kh + kv;
    P.vh = P.kl + kv;
    P.vl = P.vh + kv;
    P.inv_sk = reinterpret_cast<float *>(P.vl + kv);
    P.inv_sv = P.inv_sk + (size_t)p.n_kv * Lp;
    return P;
}

template <int HD> cudaError_t launch_hd(const AttnParams &p, void *qs, void *kvs, cudaStream_t s) {
    using A = Atc<HD>;
    const cudaError_t e = ensure_dyn_smem(reinterpret_cast<const void *>(k_attn_tc<HD>), A::SMEM);
    if (e != cudaSuccess) return e;
    const int Rp = round_up(p.rows, 128), Lp = round_up(p.max_ctx, 64);
    const Planes P = planes(p, qs, kvs);
    const int qitems = p.n_head * Rp;
    launch_pdl(k_attn_split_q<HD>, dim3((qitems + 7) / 8), dim3(kSplitThreads), 0, s, p.q, p.ldq, p.rows, Rp, p.n_head,
               P.qh, P.ql, P.inv_sq);
    const dim3 kvgrid(Lp / 64, p.n_kv);
    if (p.kv_f16)
        launch_pdl(k_attn_split_kv<HD, __half>, kvgrid, dim3(kSplitThreads), 0, s, static_cast<const __half *>(p.kcache),
                   static_cast<const __half *>(p.vcache), p.max_ctx, Lp, p.rows, static_cast<const DevState *>(p.state),
                   P.kh, P.kl, P.inv_sk, P.vh, P.vl, P.inv_sv);
    else
        launch_pdl(k_attn_split_kv<HD, float>, kvgrid, dim3(kSplitThreads), 0, s, static_cast<const float *>(p.kcache),
                   static_cast<const float *>(p.vcache), p.max_ctx, Lp, p.rows, static_cast<const DevState *>(p.state),
                   P.kh, P.kl, P.inv_sk, P.vh, P.vl, P.inv_sv);
    CUtensorMap mqh, mql, mkh, mkl, mvh, mvl;
    const int64_t kv_rows = (int64_t)p.n_kv * Lp;
    if (!tma_map_f16(&mqh, P.qh, (int64_t)p.n_head * Rp, HD, A::BQ) || !tma_map_f16(&mql, P.ql, (int64_t)p.n_head * Rp, HD, A::BQ) ||
        !tma_map_f16(&mkh, P.kh, kv_rows, HD, A::BK) || !tma_map_f16(&mkl, P.kl, kv_rows, HD, A::BK) ||
        !tma_map_f16(&mvh, P.vh, (int64_t)p.n_kv * HD, Lp, HD) || !tma_map_f16(&mvl, P.vl, (int64_t)p.n_kv * HD, Lp, HD))
        return cudaErrorInvalidValue;
    AtcArgs a;
    a.out = p.out;
    a.ldo = p.ldo;
    a.inv_sq = P.inv_sq;
    a.inv_sk = P.inv_sk;
    a.inv_sv = P.inv_sv;
    a.state = p.state;
    a.err = p.err;
    a.rows = p.rows;
    a.Rp = Rp;
    a.Lp = Lp;
    a.n_head = p.n_head;
    a.n_kv = p.n_kv;
    a.window = p.window;
    k_attn_tc<HD><<<(Rp / A::BQ) * p.n_head, A::THREADS, A::SMEM, s>>>(mqh, mql, mkh, mkl, mvh, mvl, a);
    return cudaGetLastError();
}

}  // namespace

bool attention_tc_supported(const AttnParams &p) {
    if (p.rows < 2 || (p.hd != 64 && p.hd != 128) || p.n_kv < 1 || p.n_head % p.n_kv != 0) return false;
    if (p.ldq % 4 != 0 || p.ldo % 4 != 0 || (reinterpret_cast<uintptr_t>(p.out) & 15)) return false;
    return tma_encoder_available();
}

size_t attention_tc_q_bytes(const AttnParams &p) {
    const size_t Rp = round_up(p.rows, 128);
    return (size_t)p.n_head * Rp * p.hd * 2 * sizeof(__half) + (size_t)p.n_head * Rp * sizeof(float);
}

size_t attention_tc_kv_bytes(const AttnParams &p) {
    const size_t Lp = round_up(p.max_ctx, 64);
    return (size_t)p.n_kv * Lp * p.hd * 4 * sizeof(__half) + (size_t)p.n_kv * Lp * sizeof(float) +
           (size_t)p.n_kv * (Lp / 64) * 4 * sizeof(float);
}

cudaError_t launch_attention_tc(const AttnParams &p, void *qscratch, void *kvscratch, cudaStream_t s) {
    switch (p.hd) {
    case 64: return launch_hd<64>(p, qscratch, kvscratch, s);
    case 128: return launch_hd<128>(p, qscratch, kvscratch, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace syn
