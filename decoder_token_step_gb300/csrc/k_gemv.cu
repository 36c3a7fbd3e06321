// k_gemv.cu -- weight-streaming matrix-vector products of the decode step.
//
// `matmul(h, W)` of "Local inference and architectures" (synsema.dev, section "The format"), with
// weights "multiplied in f32" (section "Choosing the engine"): every weight is dequantised to its
// exact f32 value in registers and multiplied with the f32 activation; partial sums are f32.
//
// At batch size 1 the product is bound by reading W from HBM once (2 flops per weight), so the
// kernel is built around the load stream:
//   * each warp owns R rows at a time; lane l reads the 16-byte chunks l, l+32, ... of each row
//     (128-bit, coalesced, L1 no-allocate, L2 evict-first), several chunks in flight per lane;
//   * the input vector is staged once per CTA in shared memory, laid out lane-interleaved so that
//     every float4 read is bank-conflict free; R rows share each x read;
//   * an optional RMSNorm of the input is applied while staging it (fused `rms_norm` step);
//   * the epilogue adds a bias, stores or accumulates into the destination (fused `add_bias` and
//     residual `add` steps), or forms act(gate) * up for the gated feed-forward (fused
//     `matmul, silu|gelu_tanh|..., matmul, mul` steps);
//   * the grid is at most one wave of resident CTAs (a multiple of the SM count) and every CTA
//     takes a contiguous, balanced range of row groups.
#include <algorithm>
#include <map>

#include "device_common.cuh"

namespace syn {

namespace {

constexpr int kWarps = 8;          // warps per CTA
constexpr int kThreads = kWarps * 32;
constexpr int kR = 2;              // rows per warp task
constexpr int kU = 4;              // 512-byte slabs in flight per row

struct SegInfo { int first_group; };

template <int WT, bool GATE_UP>
__global__ void __launch_bounds__(kThreads) k_gemv(const GemvParams p, int groups_total) {
    constexpr int E = Chunk<WT>::E;
    extern __shared__ __align__(16) float xs[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t K = p.seg[0].W.K;
    const int chunks = (int)(p.seg[0].W.row_bytes / 16);     // 16-byte chunks per row (>= K/E)
    const int slabs = (chunks + 31) / 32;
    const int xs_len = slabs * 32 * E;

    // ---- prologue: stage x (optionally rms-normalised) in the lane-interleaved layout ----------
    float inv = 1.f;
    if (p.norm_w) {
        __shared__ float red[kWarps];
        float ss = 0.f;
        for (int64_t i = threadIdx.x; i < K; i += kThreads) {
            float v = p.x[i];
            ss = fmaf(v, v, ss);
        }
        ss = warp_sum(ss);
        if (lane == 0) red[warp] = ss;
        __syncthreads();
        float tot = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) tot += red[w];
        inv = 1.f / sqrtf(tot / (float)K + p.eps);
    }
    for (int i = threadIdx.x; i < xs_len; i += kThreads) {
        float v = 0.f;
        if (i < K) {
            v = p.x[i];
            if (p.norm_w) v = v * inv * p.norm_w[i];
        }
        const int g = i / (32 * E), rem = i % (32 * E), l = rem / E, e = rem % E;
        xs[xs_offset<E>(g, l, e)] = v;
    }
    __syncthreads();

    // ---- this CTA's contiguous range of row groups ------------------------------------------------
    const int b = blockIdx.x, nb = gridDim.x;
    const int g0 = (int)((int64_t)groups_total * b / nb), g1 = (int)((int64_t)groups_total * (b + 1) / nb);

    for (int grp = g0 + warp; grp < g1; grp += kWarps) {
        // locate the rows of this group
        const uint8_t *rp[kR];
        const uint16_t *sp[kR];
        bool valid[kR];
        int seg = 0, row0 = grp;
        if (GATE_UP) {
            // group n = (gate row n, up row n)
#pragma unroll
            for (int r = 0; r < kR; ++r) {
                const DevMatrix &W = p.seg[r].W;
                valid[r] = true;
                rp[r] = reinterpret_cast<const uint8_t *>(W.codes) + (size_t)grp * W.row_bytes;
                sp[r] = W.scales ? W.scales + (size_t)grp * (W.K / 32) : nullptr;
            }
        } else {
            int acc_groups = 0;
            for (int s = 0; s < p.nseg; ++s) {
                int ng = (int)((p.seg[s].W.N + kR - 1) / kR);
                if (grp < acc_groups + ng) { seg = s; row0 = (grp - acc_groups) * kR; break; }
                acc_groups += ng;
            }
            const DevMatrix &W = p.seg[seg].W;
#pragma unroll
            for (int r = 0; r < kR; ++r) {
                valid[r] = row0 + r < W.N;
                int row = valid[r] ? row0 + r : row0;
                rp[r] = reinterpret_cast<const uint8_t *>(W.codes) + (size_t)row * W.row_bytes;
                sp[r] = W.scales ? W.scales + (size_t)row * (W.K / 32) : nullptr;
            }
        }

        float acc[kR];
#pragma unroll
        for (int r = 0; r < kR; ++r) acc[r] = 0.f;

        for (int s0 = 0; s0 < slabs; s0 += kU) {
            uint4 w[kU][kR];
            float sc[kU][kR];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int c = (s0 + u) * 32 + lane;
                const bool in = (s0 + u) < slabs && c < chunks;
#pragma unroll
                for (int r = 0; r < kR; ++r) {
                    w[u][r] = make_uint4(0, 0, 0, 0);
                    sc[u][r] = 0.f;
                    if (in && valid[r]) {
                        w[u][r] = ld_stream16(rp[r] + (size_t)c * 16);
                        if (WT == W_Q8_0) sc[u][r] = half_bits_to_float(ld_stream2(sp[r] + (c >> 1)));
                        if (WT == W_Q4_0) sc[u][r] = half_bits_to_float(ld_stream2(sp[r] + c));
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                if (s0 + u >= slabs) break;
                const float *xp = xs + (s0 + u) * 32 * E + lane * 4;
#pragma unroll
                for (int r = 0; r < kR; ++r) {
                    float d = Chunk<WT>::dot(w[u][r], xp);
                    if (WT == W_Q8_0 || WT == W_Q4_0)
                        acc[r] = fmaf(sc[u][r], d, acc[r]);
                    else
                        acc[r] += d;
                }
            }
        }
#pragma unroll
        for (int r = 0; r < kR; ++r) acc[r] = warp_sum(acc[r]);

        if (lane == 0) {
            if (GATE_UP) {
                float gv = acc[0], uv = acc[1];
                if (p.seg[0].bias) gv += p.seg[0].bias[grp];
                if (p.seg[1].bias) uv += p.seg[1].bias[grp];
                p.seg[0].out[grp] = apply_act(p.act, gv) * uv;
            } else {
                const GemvSeg &S = p.seg[seg];
#pragma unroll
                for (int r = 0; r < kR; ++r) {
                    if (!valid[r]) continue;
                    float y = acc[r];
                    if (S.bias) y += S.bias[row0 + r];
                    if (S.epi == EPI_ADD) y += S.out[row0 + r];
                    S.out[row0 + r] = y;
                }
            }
        }
    }
}

template <int WT, bool GU> size_t smem_bytes(int64_t row_bytes) {
    const int chunks = (int)(row_bytes / 16);
    const int slabs = (chunks + 31) / 32;
    return (size_t)slabs * 32 * Chunk<WT>::E * sizeof(float);
}

template <int WT, bool GU> void launch_t(const GemvParams &p, int sm_count, cudaStream_t s) {
    static bool attr_set = false;
    if (!attr_set) {
        // the largest dynamic allocation the device allows next to the kernel's static shared memory
        int dev = 0, optin = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        cudaFuncAttributes fa;
        cudaFuncGetAttributes(&fa, k_gemv<WT, GU>);
        cudaFuncSetAttribute(k_gemv<WT, GU>, cudaFuncAttributeMaxDynamicSharedMemorySize, optin - (int)fa.sharedSizeBytes);
        attr_set = true;
    }
    int groups = 0;
    if (GU) {
        groups = (int)p.seg[0].W.N;
    } else {
        for (int i = 0; i < p.nseg; ++i) groups += (int)((p.seg[i].W.N + kR - 1) / kR);
    }
    const size_t smem = smem_bytes<WT, GU>(p.seg[0].W.row_bytes);
    // occupancy per shared-memory size, computed once (outside any graph capture: the first
    // forward of a model always runs eagerly)
    static std::map<size_t, int> occ;
    auto it = occ.find(smem);
    if (it == occ.end()) {
        int v = 0;
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, k_gemv<WT, GU>, kThreads, smem);
        it = occ.emplace(smem, v).first;
    }
    int per_sm = it->second;
    per_sm = std::max(1, std::min(per_sm, 2));
    int blocks = std::min((groups + kWarps - 1) / kWarps, sm_count * per_sm);
    blocks = std::max(blocks, 1);
    k_gemv<WT, GU><<<blocks, kThreads, smem, s>>>(p, groups);
}

}  // namespace

void launch_gemv(const GemvParams &p, int sm_count, cudaStream_t s) {
    const int wt = p.seg[0].W.wtype;
    if (p.gate_up) {
        switch (wt) {
        case W_F32: return launch_t<W_F32, true>(p, sm_count, s);
        case W_F16: return launch_t<W_F16, true>(p, sm_count, s);
        case W_Q8_0: return launch_t<W_Q8_0, true>(p, sm_count, s);
        case W_Q4_0: return launch_t<W_Q4_0, true>(p, sm_count, s);
        }
    } else {
        switch (wt) {
        case W_F32: return launch_t<W_F32, false>(p, sm_count, s);
        case W_F16: return launch_t<W_F16, false>(p, sm_count, s);
        case W_Q8_0: return launch_t<W_Q8_0, false>(p, sm_count, s);
        case W_Q4_0: return launch_t<W_Q4_0, false>(p, sm_count, s);
        }
    }
}

// ---------------------------------------------------------------------------------------------
// Bulk rows (prefill on CUDA cores): Y[m][j] = epi(sum_k W[j][k] X[m][k]) for M input rows.
// Tiles of 32 rows x 64 outputs x 32 k; W is dequantised into shared memory tile by tile.
// ---------------------------------------------------------------------------------------------
namespace {

constexpr int GM = 32, GN = 64, GK = 32;

__global__ void __launch_bounds__(256) k_gemm_rows(const GemvParams p, int seg_idx, int64_t n_off) {
    const GemvSeg &S = p.seg[seg_idx];
    const DevMatrix &W = S.W;
    __shared__ float Xs[GM][GK + 1];
    __shared__ float Ws[GN][GK + 1];
    const int tid = threadIdx.x;
    const int m0 = blockIdx.y * GM;
    const int64_t j0 = (int64_t)blockIdx.x * GN;
    const int tr = (tid / 16) * 2, tc = (tid % 16) * 4;
    float acc[2][4] = {{0, 0, 0, 0}, {0, 0, 0, 0}};
    for (int64_t k0 = 0; k0 < W.K; k0 += GK) {
        for (int i = tid; i < GM * GK; i += 256) {
            int r = i / GK, kk = i % GK;
            int m = m0 + r;
            int64_t k = k0 + kk;
            Xs[r][kk] = (m < p.rows && k < W.K) ? p.x[(size_t)m * p.ldx + k] : 0.f;
        }
        for (int i = tid; i < GN * GK; i += 256) {
            int r = i / GK, kk = i % GK;
            int64_t j = j0 + r, k = k0 + kk;
            Ws[r][kk] = (j < W.N && k < W.K) ? dequant_one(W, j, k) : 0.f;
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < GK; ++kk) {
            float a0 = Xs[tr][kk], a1 = Xs[tr + 1][kk];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                float b = Ws[tc + c][kk];
                acc[0][c] = fmaf(a0, b, acc[0][c]);
                acc[1][c] = fmaf(a1, b, acc[1][c]);
            }
        }
        __syncthreads();
    }
    for (int r = 0; r < 2; ++r) {
        int m = m0 + tr + r;
        if (m >= p.rows) continue;
        for (int c = 0; c < 4; ++c) {
            int64_t j = j0 + tc + c;
            if (j >= W.N) continue;
            float y = acc[r][c];
            if (S.bias) y += S.bias[j];
            float *o = S.out + (size_t)m * S.ldo + j;
            if (S.epi == EPI_ADD) y += *o;
            *o = y;
        }
    }
    (void)n_off;
}

}  // namespace

void launch_gemm_rows(const GemvParams &p, cudaStream_t s) {
    for (int i = 0; i < p.nseg; ++i) {
        dim3 grid((unsigned)((p.seg[i].W.N + GN - 1) / GN), (unsigned)((p.rows + GM - 1) / GM));
        k_gemm_rows<<<grid, 256, 0, s>>>(p, i, 0);
    }
}

int gemv_max_blocks_per_sm(int wtype, int64_t K, int gate_up) {
    (void)wtype; (void)K; (void)gate_up;
    return 2;
}

}  // namespace syn
