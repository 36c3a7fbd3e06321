// k_gemv.cu -- the standalone weight-streaming GEMV kernel (one launch per fused matmul node; the
// device code is in gemv_dev.cuh) and the CUDA-core GEMM used by bulk prefill when the tensor-core
// path does not apply.
#include <algorithm>

#include "gemv_dev.cuh"

namespace syn {

namespace {

// KR rows per warp task, KU 32-byte chunks per row and batch, NW warps: one CTA per SM (16 warps
// at up to 128 registers fill the register file). Two layouts (launch_w): KR = 1, KU = 4 -- a
// 4096-byte row is one batch per lane, issued at once, so the short matmuls of a decode step
// (Q/K/V, the output projection, the down projection) keep twice the bytes in flight from their
// first instruction -- and KR = 2, KU = 2 for the gate/up pairs, for matrices of many rows (the
// logits) and for many rows of at most 2 KB. Q4_0's two-row forms run 8 warps (their registers).
template <int WT, bool GATE_UP, int KR, int KU, int NW>
__global__ void __launch_bounds__(NW * 32, 1) k_gemv(const GemvParams p, int groups_total) {
    extern __shared__ __align__(16) float xs[];
    __shared__ float red[NW];
    gemv_cta<WT, GATE_UP, KR, KU, NW, false>(p, GemvPre{}, groups_total, blockIdx.x, gridDim.x, xs, red, [] {
        pdl_launch_dependents();
        pdl_wait();
    });
}

// the same with a post-branch update of x in the prologue (GemvPre)
template <int WT, bool GATE_UP, int KR, int KU, int NW>
__global__ void __launch_bounds__(NW * 32, 1) k_gemv_pre(const GemvParams p, const GemvPre pre, int groups_total) {
    extern __shared__ __align__(16) float xs[];
    __shared__ float red[NW];
    gemv_cta<WT, GATE_UP, KR, KU, NW, true>(p, pre, groups_total, blockIdx.x, gridDim.x, xs, red, [] {
        pdl_launch_dependents();
        pdl_wait();
    });
}

template <int WT, bool GU, int KR, int KU, int NW> void launch_t(GemvParams p, int sm_count, cudaStream_t s, const GemvPre *pre) {
    gemv_set_groups(p, KR);
    const int groups = gemv_groups(p, KR);
    const size_t smem = gemv_smem_bytes<WT>(p.seg[0].W.row_bytes);
    const int blocks = std::max(1, std::min((groups + NW - 1) / NW, sm_count));
    // a failure of ensure_dyn_smem makes the launch below fail, and that error reaches the caller
    if (pre) {
        auto *fn = k_gemv_pre<WT, GU, KR, KU, NW>;
        ensure_dyn_smem(reinterpret_cast<const void *>(fn), (int)smem);
        launch_pdl(fn, dim3(blocks), dim3(NW * 32), smem, s, p, *pre, groups);
    } else {
        auto *fn = k_gemv<WT, GU, KR, KU, NW>;
        ensure_dyn_smem(reinterpret_cast<const void *>(fn), (int)smem);
        launch_pdl(fn, dim3(blocks), dim3(NW * 32), smem, s, p, groups);
    }
}

// many rows: the two-row layout streams the logits matrix faster
constexpr int64_t kGemvManyRows = 65536;

template <int WT> void launch_w(const GemvParams &p, int sm_count, cudaStream_t s, const GemvPre *pre) {
    // the Q4_0 decode of two rows needs more than the 128 registers a thread has at 16 warps
    constexpr int NW2 = WT == W_Q4_0 ? 8 : 16;
    int64_t rows = 0;
    for (int i = 0; i < p.nseg; ++i) rows += p.seg[i].W.N;
    if (p.gate_up) return launch_t<WT, true, 2, 2, NW2>(p, sm_count, s, pre);
    // rows of at most two 32-lane slabs of chunks (2 KB) fill only half a lane's four-chunk batch:
    // when one-row tasks would take more than one round of the warps, two rows a task issue every
    // row at once (not for Q4_0, whose two-row form runs at 8 warps)
    const bool short_rows = WT != W_Q4_0 && p.seg[0].W.row_bytes <= 2048 && rows > (int64_t)16 * sm_count;
    if (rows >= kGemvManyRows || short_rows) return launch_t<WT, false, 2, 2, NW2>(p, sm_count, s, pre);
    return launch_t<WT, false, 1, 4, 16>(p, sm_count, s, pre);
}

}  // namespace

void launch_gemv(const GemvParams &p, int sm_count, cudaStream_t s, const GemvPre *pre) {
    switch (p.seg[0].W.wtype) {
    case W_F32: return launch_w<W_F32>(p, sm_count, s, pre);
    case W_F16: return launch_w<W_F16>(p, sm_count, s, pre);
    case W_Q8_0: return launch_w<W_Q8_0>(p, sm_count, s, pre);
    case W_Q4_0: return launch_w<W_Q4_0>(p, sm_count, s, pre);
    }
}

// ---------------------------------------------------------------------------------------------
// Bulk rows (prefill on CUDA cores): Y[m][j] = epi(sum_k W[j][k] X[m][k]) for M input rows.
// Tiles of 32 rows x 64 outputs x 32 k; W is dequantised into shared memory tile by tile.
// ---------------------------------------------------------------------------------------------
namespace {

constexpr int GM = 32, GN = 64, GK = 32;

__global__ void __launch_bounds__(256) k_gemm_rows(const GemvParams p, int seg_idx) {
    const GemvSeg &S = p.seg[seg_idx];
    const DevMatrix &W = S.W;
    __shared__ float Xs[GM][GK + 1];
    __shared__ float Ws[GN][GK + 1];
    const int tid = threadIdx.x;
    const int m0 = blockIdx.y * GM;
    const int64_t j0 = (int64_t)blockIdx.x * GN;
    const int tr = (tid / 16) * 2, tc = (tid % 16) * 4;
    float acc[2][4] = {{0, 0, 0, 0}, {0, 0, 0, 0}};
    pdl_wait();
    for (int64_t k0 = 0; k0 < W.K; k0 += GK) {
        for (int i = tid; i < GM * GK; i += 256) {
            const int r = i / GK, kk = i % GK;
            const int m = m0 + r;
            const int64_t k = k0 + kk;
            Xs[r][kk] = (m < p.rows && k < W.K) ? p.x[(size_t)m * p.ldx + k] : 0.f;
        }
        for (int i = tid; i < GN * GK; i += 256) {
            const int r = i / GK, kk = i % GK;
            const int64_t j = j0 + r, k = k0 + kk;
            Ws[r][kk] = (j < W.N && k < W.K) ? dequant_one(W, j, k) : 0.f;
        }
        __syncthreads();
#pragma unroll 8
        for (int kk = 0; kk < GK; ++kk) {
            const float a0 = Xs[tr][kk], a1 = Xs[tr + 1][kk];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const float bv = Ws[tc + c][kk];
                acc[0][c] = fmaf(a0, bv, acc[0][c]);
                acc[1][c] = fmaf(a1, bv, acc[1][c]);
            }
        }
        __syncthreads();
    }
    for (int r = 0; r < 2; ++r) {
        const int m = m0 + tr + r;
        if (m >= p.rows) continue;
        for (int c = 0; c < 4; ++c) {
            const int64_t j = j0 + tc + c;
            if (j >= W.N) continue;
            float y = acc[r][c];
            if (S.bias) y += S.bias[j];
            float *o = S.out + (size_t)m * S.ldo + j;
            if (S.epi == EPI_ADD) y += *o;
            *o = y;
        }
    }
}

}  // namespace

void launch_gemm_rows(const GemvParams &p, cudaStream_t s) {
    for (int i = 0; i < p.nseg; ++i) {
        dim3 grid((unsigned)((p.seg[i].W.N + GN - 1) / GN), (unsigned)((p.rows + GM - 1) / GM));
        launch_pdl(k_gemm_rows, grid, dim3(256), 0, s, p, i);
    }
}

}  // namespace syn
