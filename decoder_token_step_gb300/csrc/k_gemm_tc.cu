// k_gemm_tc.cu -- bulk-prefill matmuls on the 5th-generation tensor cores (tcgen05, TMEM, TMA).
//
// Bulk prefill runs every matmul of the block over n prompt rows at once ("Execution contract",
// section "Prefill": the whole prompt in one forward, then `last`), so Y[m][j] = sum_k W[j][k] X[m][k]
// is a dense GEMM of n x K by K x N. The decoder multiplies weights in f32 ("Local inference and
// architectures", section "Choosing the engine"), so the tensor cores get an f32-accurate split.
// Every row r of X and of W is scaled by a power of two s_r that puts its largest magnitude just
// under 2^14 (inside the f16 range, exactly undone later), then split into two f16 halves:
//     w s = wh + wl,  x s' = xh + xl      (wh = f16(w s), wl = f16(w s - wh); same for x)
//     w x ~= (wh xh + wh xl + wl xh) / (s s')
// Each half carries 11 significant bits, so the split keeps 22 and the dropped wl xl term is near
// 2^-22 of the product: three f16 MMAs give an f32-grade dot product. (A bf16 split keeps only 16
// bits; measured on llama-3-8B shapes its prompt logits drift ~4x further from the f32 oracle than
// an f32 CUDA-core GEMM's.) f16 weights are exact in wh alone.
//
// Three kernels per matmul node:
//   k_split_rows     X (f32, n rows) -> Xh, Xl (f16 [n][K]) + 1/s' per row, once per node
//   k_dequant_split  W (GGUF storage) -> Wh, Wl (f16 [N][K]) + 1/s per row, into a scratch buffer
//                    (skipped when the weight's planes are kept resident, option tc_planes)
//   k_gemm_tc        output tiles of 128 weight rows x BN prompt rows (BN = 256, or 128 when the
//                    matmul has too few tiles to fill whole waves with the wide tile), one
//                    persistent CTA per SM walking tiles b, b + G, ...; the stage ring, the MMA
//                    stream and the drain chain run on across tile boundaries, so a tile's stores
//                    overlap the next tile's loads and MMAs:
//       warp 0        TMA producer: per 64-wide K slice, four tiles (Wh, Wl: 16 KB each; Xh, Xl:
//                     BN x 128 bytes each) with the 128-byte swizzle into a shared-memory ring (2
//                     stages of 96 KB for BN = 256, 3 stages of 64 KB for BN = 128), completion on
//                     an mbarrier;
//       warp 1        allocates all 512 TMEM columns (512 / BN f32 accumulators of 128 lanes x BN);
//                     one thread issues 12 tcgen05.mma (kind::f16, M = 128, N = BN, K = 16) per
//                     slice, eight slices per accumulator before moving to the next, and commits
//                     every stage back to the producer;
//       warps 2..    BN / 32 epilogue warps, two per TMEM lane quadrant for BN = 256 (128
//                     accumulator columns each): per eight slices, tcgen05.ld of the accumulator
//                     (TMEM lane = weight row) added into f32 registers, then the buffer is handed
//                     back; at the tile's end bias, store or accumulate into Y (32 lanes write 32
//                     consecutive outputs).
// Why drain at all: the tensor core's f32 accumulation is not rounded to nearest (measured: over
// K = 14336 in one accumulator the error grows faster than sqrt(K) and leans toward zero), and the
// decoder's deep residual stream amplifies such a drift; summing 512-wide partial products in
// registers keeps the matmul close to an f32 dot product (llama-3-8B at full size, 16-token bulk
// prompt: 1.5e-4 relative logit error; 7e-5 when draining every 128 products, which costs 14 %
// more time). Several accumulators let the MMA thread run ahead of the epilogue.
// Tile order: prompt-row tiles fastest, then weight-row tiles, so the CTAs that run together share
// one weight tile in L2 and each weight tile leaves HBM once.
//
// Every wait is bounded: a wait that runs out sets ERR_TC in the device state, and the CTA still
// waits (bounded) for its committed MMAs before it frees its TMEM and returns.
#include <cuda.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "tc_dev.cuh"

namespace syn {

namespace {

constexpr int TC_BM = 128;                        // weight rows per tile (MMA M)
constexpr int TC_BK = 64;                         // K per stage: one 128-byte swizzle row of f16
constexpr int TC_TILE_W = TC_BM * TC_BK * 2;      // bytes of one f16 weight tile
constexpr int TC_DRAIN = 8;                       // K slices (512 products) accumulated in TMEM between drains

// Tile shapes. BN prompt rows per tile (MMA N): 256 reads 96 KB per 64-wide K slice for a
// 128 x 256 output tile (7.6 KB per MFLOP of tensor work), 128 reads 64 KB for 128 x 128 (10.2 KB
// per MFLOP); the bytes each SM must take in per flop are what bounds this kernel.
template <int BN> struct TcCfg {
    static constexpr int TILE_X = BN * TC_BK * 2;             // bytes of one f16 activation tile
    static constexpr int STAGE = 2 * TC_TILE_W + 2 * TILE_X;
    static constexpr int STAGES = BN == 256 ? 2 : 3;
    static constexpr int SMEM = STAGES * STAGE + 1024;        // + slack to align the ring to 1024 bytes
    static constexpr int NBUF = 512 / BN;                     // f32 accumulators of 128 lanes x BN columns
    static constexpr int TMEM_COLS = NBUF * BN;               // all 512 columns of the SM
    static constexpr int EW = BN / 32;                        // epilogue warps: 4 lane quadrants x BN/128 halves
    static constexpr int THREADS = 64 + 32 * EW;
};

// One output matrix of a launch: the launch walks the tiles of all its segments (matmuls on the
// same input: Q/K/V, gate and up) as one tile space, segment by segment.
struct TcSeg {
    float *out;
    int64_t ldo;
    const float *bias;
    const float *inv_sw;   // [N] 1 / (row scale of W)
    int epi;
    int N;
    int tile0;             // first tile of this segment in the launch's tile space
};
struct TcArgs {
    TcSeg seg[3];
    int nseg;
    int ntiles;            // tiles of all segments
    const float *inv_sx;   // [M] 1 / (row scale of X)
    int M, K;
    int *err;
};


template <int BN>
__global__ void __launch_bounds__(TcCfg<BN>::THREADS, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap tWh0, const __grid_constant__ CUtensorMap tWl0,
              const __grid_constant__ CUtensorMap tWh1, const __grid_constant__ CUtensorMap tWl1,
              const __grid_constant__ CUtensorMap tWh2, const __grid_constant__ CUtensorMap tWl2,
              const __grid_constant__ CUtensorMap tXh, const __grid_constant__ CUtensorMap tXl, const TcArgs a) {
    using C = TcCfg<BN>;
    constexpr int TC_STAGES = C::STAGES, TC_STAGE = C::STAGE, TC_TILE_X = C::TILE_X, TC_NBUF = C::NBUF;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *ring = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    __shared__ __align__(8) uint64_t full[TC_STAGES], empty[TC_STAGES], acc_full[TC_NBUF], acc_empty[TC_NBUF], done;
    __shared__ uint32_t tmem_base;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // persistent: tiles b, b + G, ... with b the CTA index and G the grid size
    const int mg = (a.M + BN - 1) / BN, ntiles = a.ntiles;
    const int u0 = blockIdx.x, ustep = gridDim.x;
    // tile t: segment, then (prompt-row group lt % mg, weight-row tile lt / mg) inside it
    auto seg_of = [&](int t) { return (a.nseg > 1 && t >= a.seg[1].tile0) + (a.nseg > 2 && t >= a.seg[2].tile0); };
    auto m0_of = [&](int lt) { return (lt % mg) * BN; };
    const int nk = (a.K + TC_BK - 1) / TC_BK;
    const int nchunks = (nk + TC_DRAIN - 1) / TC_DRAIN;   // per tile

    if (threadIdx.x == 0) {
        for (int s = 0; s < TC_STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);   // the MMA commit
        }
        for (int b = 0; b < TC_NBUF; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], C::EW);   // one arrival per epilogue warp
        }
        mbar_init(&done, 1);
        mbar_init_fence();
    }
    if (warp == 1) {
        tmem_alloc(&tmem_base, C::TMEM_COLS);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;

    if (warp == 0) {
        if (lane == 0) {
            // stage counter g runs across tiles: the ring never drains between tiles
            int g = 0;
            bool ok = true;
            for (int t = u0; t < ntiles && ok; t += ustep) {
                const int sg = seg_of(t), lt = t - a.seg[sg].tile0;
                const int m0 = m0_of(lt), n0 = (lt / mg) * TC_BM;
                const CUtensorMap *mwh = sg == 0 ? &tWh0 : (sg == 1 ? &tWh1 : &tWh2);
                const CUtensorMap *mwl = sg == 0 ? &tWl0 : (sg == 1 ? &tWl1 : &tWl2);
                for (int kb = 0; kb < nk; ++kb, ++g) {
                    const int s = g % TC_STAGES;
                    if (g >= TC_STAGES && !mbar_wait(&empty[s], ((g / TC_STAGES) - 1) & 1, a.err, ERR_TC)) {
                        ok = false;
                        break;
                    }
                    uint8_t *st = ring + s * TC_STAGE;
                    mbar_expect_tx(&full[s], TC_STAGE);
                    tma_load_2d(st, mwh, kb * TC_BK, n0, &full[s]);
                    tma_load_2d(st + TC_TILE_W, mwl, kb * TC_BK, n0, &full[s]);
                    tma_load_2d(st + 2 * TC_TILE_W, &tXh, kb * TC_BK, m0, &full[s]);
                    tma_load_2d(st + 2 * TC_TILE_W + TC_TILE_X, &tXl, kb * TC_BK, m0, &full[s]);
                }
            }
            // nothing may land in shared memory once the CTA has gone: wait for the stages in flight
            for (int g2 = max(0, g - TC_STAGES); g2 < g; ++g2) mbar_wait(&full[g2 % TC_STAGES], (g2 / TC_STAGES) & 1, a.err, ERR_TC);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = tc_idesc_f16(TC_BM, BN);
            int g = 0, c = 0;   // global stage and chunk counters
            bool ok = true;
            for (int t = u0; t < ntiles && ok; t += ustep) {
                for (int kb = 0; kb < nk; ++kb, ++g) {
                    const int s = g % TC_STAGES, b = c % TC_NBUF;
                    const bool first = kb % TC_DRAIN == 0, last = kb % TC_DRAIN == TC_DRAIN - 1 || kb == nk - 1;
                    // a chunk's accumulator buffer must have been drained by the epilogue
                    if (first && c >= TC_NBUF && !mbar_wait(&acc_empty[b], ((c / TC_NBUF) - 1) & 1, a.err, ERR_TC)) {
                        ok = false;
                        break;
                    }
                    if (!mbar_wait(&full[s], (g / TC_STAGES) & 1, a.err, ERR_TC)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t base = saddr(ring + s * TC_STAGE);
                    const uint32_t wh = base, wl = base + TC_TILE_W, xh = base + 2 * TC_TILE_W, xl = xh + TC_TILE_X;
                    const uint32_t d = tmem + (uint32_t)(b * BN);
#pragma unroll
                    for (int k = 0; k < TC_BK / 16; ++k) {
                        const uint32_t off = k * 32;   // 16 halves along K inside the swizzled row
                        mma_f16(d, desc_sw128(wh + off), desc_sw128(xh + off), idesc, !first || k != 0);
                        mma_f16(d, desc_sw128(wh + off), desc_sw128(xl + off), idesc, 1);
                        mma_f16(d, desc_sw128(wl + off), desc_sw128(xh + off), idesc, 1);
                    }
                    // the stage is free once these MMAs have read it
                    mma_commit(&empty[s]);
                    if (last) {
                        mma_commit(&acc_full[b]);           // the chunk's partial product is complete
                        ++c;
                    }
                }
            }
            mma_commit(&done);              // arrives when every MMA issued above has completed
        }
    } else {
        // epilogue: warp w owns TMEM lanes 32 * (w % 4) .. + 31, i.e. weight rows n0 + that, and
        // accumulator columns hf * 128 .. + 127 (prompt rows m0 + that), hf = (w - 2) / 4. Each
        // chunk of TC_DRAIN 64-wide K slices is accumulated by the tensor core into a fresh buffer
        // and added here in f32 with round-to-nearest, so the tensor core's own accumulation never
        // runs over more than 12 * TC_DRAIN products of 16 terms. While it stores a finished tile,
        // the MMA thread already fills the next buffers with the next tile's first chunks.
        const int q = warp & 3, hf = (warp - 2) >> 2;
        bool ok = true;
        int c = 0;
        for (int t = u0; t < ntiles && ok; t += ustep) {
            const int sg = seg_of(t), lt = t - a.seg[sg].tile0;
            const TcSeg &S = a.seg[sg];
            const int m0 = m0_of(lt) + hf * 128, n0 = (lt / mg) * TC_BM;
            const int n = n0 + q * 32 + lane;
            float acc[128];
#pragma unroll
            for (int j = 0; j < 128; ++j) acc[j] = 0.f;
            for (int cc = 0; cc < nchunks; ++cc, ++c) {
                const int b = c % TC_NBUF;
                ok = mbar_wait(&acc_full[b], (c / TC_NBUF) & 1, a.err, ERR_TC);
                if (!ok) break;
                tc_fence_after();
                const uint32_t tt = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(b * BN + hf * 128);
#pragma unroll
                for (int c0 = 0; c0 < 128; c0 += 32) {
                    uint32_t r[32];
                    tmem_ld32(tt + (uint32_t)c0, r);
#pragma unroll
                    for (int j = 0; j < 32; ++j) acc[c0 + j] += __uint_as_float(r[j]);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acc_empty[b]);
            }
            if (ok && n < S.N) {
                const float bias = S.bias ? S.bias[n] : 0.f;
                const float sw = S.inv_sw[n];
                // ST rows at a time: the residual reads of a group are issued together, ahead of
                // its stores (lanes write 32 consecutive outputs of one row)
                constexpr int ST = BN == 256 ? 8 : 16;
#pragma unroll
                for (int j0 = 0; j0 < 128; j0 += ST) {
                    float prev[ST], sx[ST];
#pragma unroll
                    for (int j = 0; j < ST; ++j) {
                        const int m = m0 + j0 + j;
                        prev[j] = (S.epi == EPI_ADD && m < a.M) ? __ldcg(S.out + (size_t)m * S.ldo + n) : 0.f;
                        sx[j] = m < a.M ? a.inv_sx[m] : 0.f;
                    }
#pragma unroll
                    for (int j = 0; j < ST; ++j) {
                        const int m = m0 + j0 + j;
                        if (m < a.M) S.out[(size_t)m * S.ldo + n] = prev[j] + (acc[j0 + j] * sx[j] * sw + bias);   // exact: powers of two
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        // the columns are freed only after every committed MMA has finished writing them
        if (lane == 0) mbar_wait(&done, 0, a.err, ERR_TC);
        __syncwarp();
        tc_fence_after();
        tmem_free(tmem, C::TMEM_COLS);
    }
}

SYN_DEV float block_max(float v, float *red) {
    v = warp_max(v);
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    __syncthreads();
    if (lane == 0) red[w] = v;
    __syncthreads();
    float m = 0.f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) m = fmaxf(m, red[i]);
    return m;
}

// X (f32 rows, stride ldx) -> scaled hi/lo f16 planes [M][K] and 1/scale per row; one CTA per row
__global__ void k_split_rows(const float *x, int64_t ldx, int M, int K, __half *xh, __half *xl, float *inv_s) {
    __shared__ float red[32];
    pdl_wait();
    for (int m = blockIdx.x; m < M; m += gridDim.x) {
        const float *row = x + (size_t)m * ldx;
        float amax = 0.f;
        for (int k = threadIdx.x * 4; k < K; k += blockDim.x * 4) {
            const float4 v = *reinterpret_cast<const float4 *>(row + k);
            amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
        }
        const float sc = row_scale(block_max(amax, red));
        if (threadIdx.x == 0) inv_s[m] = 1.f / sc;
        for (int k = threadIdx.x * 4; k < K; k += blockDim.x * 4) {
            const float4 v = *reinterpret_cast<const float4 *>(row + k);
            const float f[4] = {v.x * sc, v.y * sc, v.z * sc, v.w * sc};
            __half h[4], l[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) split2(f[e], h[e], l[e]);
            *reinterpret_cast<uint2 *>(xh + (size_t)m * K + k) = *reinterpret_cast<const uint2 *>(h);
            *reinterpret_cast<uint2 *>(xl + (size_t)m * K + k) = *reinterpret_cast<const uint2 *>(l);
        }
    }
}

// The 8 dequantised values W[row][k0 .. k0+7] (k0 a multiple of 8) from one vector load.
SYN_DEV void dequant8(const DevMatrix &W, int64_t row, int64_t k0, float (&v)[8]) {
    const uint8_t *rp = static_cast<const uint8_t *>(W.codes) + (size_t)row * W.row_bytes;
    switch (W.wtype) {
    case W_F32: {
        const float4 a = __ldg(reinterpret_cast<const float4 *>(rp) + k0 / 4);
        const float4 b = __ldg(reinterpret_cast<const float4 *>(rp) + k0 / 4 + 1);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
        return;
    }
    case W_F16: {
        const uint4 c = __ldg(reinterpret_cast<const uint4 *>(rp + k0 * 2));
        const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w[i]));
            v[2 * i] = f.x;
            v[2 * i + 1] = f.y;
        }
        return;
    }
    case W_Q8_0: {
        // offset-binary codes (q + 128)
        const float d = half_bits_to_float(__ldg(W.scales + (size_t)row * W.scale_stride + k0 / 32));
        const uint2 c = __ldg(reinterpret_cast<const uint2 *>(rp + k0));
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[i] = d * (float)((int)((c.x >> (8 * i)) & 255u) - 128);
            v[4 + i] = d * (float)((int)((c.y >> (8 * i)) & 255u) - 128);
        }
        return;
    }
    case W_Q4_0: {
        // block b: element j < 16 is the low nibble of byte j, element j >= 16 the high nibble of byte j - 16
        const int64_t b = k0 / 32, j0 = k0 % 32;
        const float d = half_bits_to_float(__ldg(W.scales + (size_t)row * W.scale_stride + b));
        const uint2 c = __ldg(reinterpret_cast<const uint2 *>(rp + b * 16 + (j0 & 15)));
        const int sh = j0 < 16 ? 0 : 4;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[i] = d * (float)((int)((c.x >> (8 * i + sh)) & 15u) - 8);
            v[4 + i] = d * (float)((int)((c.y >> (8 * i + sh)) & 15u) - 8);
        }
        return;
    }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = 0.f;
}

// W (any storage type) -> scaled hi/lo f16 planes [N][K] and 1/scale per row; one CTA per row,
// 8 consecutive elements per thread step (one vector load), two passes (row maximum, then split)
__global__ void k_dequant_split(const DevMatrix W, __half *wh, __half *wl, float *inv_s) {
    __shared__ float red[32];
    const int64_t K = W.K;
    pdl_wait();
    for (int64_t j = blockIdx.x; j < W.N; j += gridDim.x) {
        float amax = 0.f;
        for (int64_t k = threadIdx.x * 8; k < K; k += blockDim.x * 8) {
            float v[8];
            dequant8(W, j, k, v);
#pragma unroll
            for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(v[e]));
        }
        const float sc = row_scale(block_max(amax, red));
        if (threadIdx.x == 0) inv_s[j] = 1.f / sc;
        for (int64_t k = threadIdx.x * 8; k < K; k += blockDim.x * 8) {
            float v[8];
            dequant8(W, j, k, v);
            __half h[8], l[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) split2(v[e] * sc, h[e], l[e]);
            *reinterpret_cast<uint4 *>(wh + j * K + k) = *reinterpret_cast<const uint4 *>(h);
            *reinterpret_cast<uint4 *>(wl + j * K + k) = *reinterpret_cast<const uint4 *>(l);
        }
    }
}

using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                 const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encoder() {
    static EncodeTiled fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiled>(p);
    });
    return fn;
}

// SMs of the current device
int sm_count() {
    int dev = 0, v = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    return v > 0 ? v : 148;
}

}  // namespace

bool tma_encoder_available() { return encoder() != nullptr; }

bool tma_map_f16(CUtensorMap *map, const void *base, int64_t rows, int64_t cols, int box_rows) {
    EncodeTiled enc = encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool gemm_tc_supported(const GemvParams &p) {
    if (p.norm_w || p.gate_up || p.rows < 1) return false;
    const int64_t K = p.seg[0].W.K;
    if (K % 8 != 0 || p.ldx % 4 != 0 || (reinterpret_cast<uintptr_t>(p.x) & 15)) return false;
    for (int i = 0; i < p.nseg; ++i)
        if (p.seg[i].W.K != K) return false;
    return encoder() != nullptr;
}

// scratch layout: [hi plane][lo plane][1/scale per row]
size_t gemm_tc_x_bytes(const GemvParams &p) {
    return (size_t)p.rows * p.seg[0].W.K * 2 * sizeof(__half) + (size_t)p.rows * sizeof(float);
}

// every segment's planes at once (one launch walks all segments), each 256-byte aligned
size_t gemm_tc_w_bytes(const GemvParams &p) {
    size_t b = 0;
    for (int i = 0; i < p.nseg; ++i)
        b += ((size_t)p.seg[i].W.N * p.seg[i].W.K * 2 * sizeof(__half) + (size_t)p.seg[i].W.N * sizeof(float) + 255) / 256 * 256;
    return b;
}

size_t gemm_tc_planes_bytes(const DevMatrix &W) {
    return (size_t)W.N * W.K * 2 * sizeof(__half) + (size_t)W.N * sizeof(float);
}

cudaError_t launch_dequant_split(const DevMatrix &W, void *planes, cudaStream_t s) {
    __half *wh = static_cast<__half *>(planes), *wl = wh + (size_t)W.N * W.K;
    float *sw = reinterpret_cast<float *>(wl + (size_t)W.N * W.K);
    k_dequant_split<<<(unsigned)std::min<int64_t>(W.N, 152 * 8), 256, 0, s>>>(W, wh, wl, sw);
    return cudaGetLastError();
}

cudaError_t launch_gemm_tc(const GemvParams &p, const void *const planes_in[3], void *xscratch, void *wscratch, int *err,
                           cudaStream_t s) {
    cudaError_t e = ensure_dyn_smem(reinterpret_cast<const void *>(k_gemm_tc<128>), TcCfg<128>::SMEM);
    if (e == cudaSuccess) e = ensure_dyn_smem(reinterpret_cast<const void *>(k_gemm_tc<256>), TcCfg<256>::SMEM);
    if (e != cudaSuccess) return e;
    const int M = p.rows;
    const int64_t K = p.seg[0].W.K;
    __half *xh = static_cast<__half *>(xscratch), *xl = xh + (size_t)M * K;
    float *sx = reinterpret_cast<float *>(xl + (size_t)M * K);
    launch_pdl(k_split_rows, dim3((unsigned)std::min(M, 152 * 8)), dim3(256), 0, s, p.x, p.ldx, M, (int)K, xh, xl, sx);
    // Tile width per node: a persistent grid walks whole waves of tiles (all segments in one tile
    // space), so pick the width whose rounds x per-tile work is smallest, counting a 128-row tile's
    // flops 15 % dearer (it reads 10.2 KB per MFLOP against 7.6 KB for 256 rows). The activation
    // maps load BN-row boxes.
    auto node_cost = [&](int bn) {
        int64_t tiles = 0;
        for (int i = 0; i < p.nseg; ++i) tiles += (M + bn - 1) / bn * ((p.seg[i].W.N + TC_BM - 1) / TC_BM);
        return (double)((tiles + sm_count() - 1) / sm_count()) * (bn == 256 ? 2.0 : 1.15);
    };
    const bool wide = M >= 256 && node_cost(256) <= node_cost(128);
    const int BN = wide ? 256 : 128;
    CUtensorMap mxh, mxl;
    if (!tma_map_f16(&mxh, xh, M, K, BN) || !tma_map_f16(&mxl, xl, M, K, BN)) return cudaErrorInvalidValue;

    TcArgs a = {};
    CUtensorMap mwh[3], mwl[3];
    uint8_t *scratch = static_cast<uint8_t *>(wscratch);
    int tiles = 0;
    for (int i = 0; i < p.nseg; ++i) {
        const GemvSeg &S = p.seg[i];
        const int64_t N = S.W.N;
        // the weight's f16 hi/lo planes: resident if built at load, else converted into scratch now
        void *planes = const_cast<void *>(planes_in[i]);
        if (!planes) {
            planes = scratch;
            scratch += (gemm_tc_planes_bytes(S.W) + 255) / 256 * 256;
        }
        __half *wh = static_cast<__half *>(planes), *wl = wh + (size_t)N * K;
        float *sw = reinterpret_cast<float *>(wl + (size_t)N * K);
        if (!planes_in[i])
            launch_pdl(k_dequant_split, dim3((unsigned)std::min<int64_t>(N, 152 * 8)), dim3(256), 0, s, S.W, wh, wl, sw);
        if (!tma_map_f16(&mwh[i], wh, N, K, TC_BM) || !tma_map_f16(&mwl[i], wl, N, K, TC_BM)) return cudaErrorInvalidValue;
        TcSeg &G = a.seg[i];
        G.out = S.out;
        G.ldo = S.ldo;
        G.bias = S.bias;
        G.inv_sw = sw;
        G.epi = S.epi;
        G.N = (int)N;
        G.tile0 = tiles;
        const int mgroups = (M + BN - 1) / BN;
        tiles += mgroups * (int)((N + TC_BM - 1) / TC_BM);
    }
    for (int i = p.nseg; i < 3; ++i) {
        mwh[i] = mwh[0];
        mwl[i] = mwl[0];
    }
    a.nseg = p.nseg;
    a.ntiles = tiles;
    a.inv_sx = sx;
    a.M = M;
    a.K = (int)K;
    a.err = err;
    if (wide) {
        k_gemm_tc<256><<<std::min(tiles, sm_count()), TcCfg<256>::THREADS, TcCfg<256>::SMEM, s>>>(
            mwh[0], mwl[0], mwh[1], mwl[1], mwh[2], mwl[2], mxh, mxl, a);
    } else {
        k_gemm_tc<128><<<std::min(tiles, sm_count()), TcCfg<128>::THREADS, TcCfg<128>::SMEM, s>>>(
            mwh[0], mwl[0], mwh[1], mwl[1], mwh[2], mwl[2], mxh, mxl, a);
    }
    return cudaGetLastError();
}

}  // namespace syn
