// k_step.cuh -- the persistent decode-step kernel: one forward at n = 1 ("Execution contract",
// section "Forward phase") as a single launch.
//
// One cooperative launch runs a whole decode step: the fused plan's nodes become phases (GEMV,
// per-head transforms, attention, norms, elementwise ops, embed, argmax) in device memory, and
// every CTA walks them in order with a grid barrier between consecutive phases. There is no launch
// gap between phases, and each phase first issues the work that does not depend on the previous one
// -- the first weight loads of a GEMV, the L2 prefetch of the old KV positions of an attention --
// and only then waits at the barrier, so HBM stays busy across phase boundaries.
//
// The barrier: every CTA's thread 0 adds 1 to a global counter (release) and polls it (acquire)
// until all CTAs of the phase have arrived. Polling is bounded: after ~0.4 s it sets ERR_BARRIER in
// the device state and the CTA stops, so a broken launch cannot hang the GPU. The cooperative
// launch guarantees that all CTAs are resident, so in a correct launch every barrier completes.
#pragma once

#include "attn_dev.cuh"
#include "gemv_dev.cuh"
#include "misc_dev.cuh"

namespace syn {

constexpr int kStepThreads = 256;
constexpr int kStepU = 2;   // GEMV chunks per row per batch
constexpr unsigned kBarrierSpins = 1u << 22;

SYN_DEV unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

SYN_DEV unsigned ld_acquire(const unsigned *p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
SYN_DEV void red_release_add(unsigned *p, unsigned v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Returns false if the barrier timed out (the error is recorded in *err).
SYN_DEV bool grid_barrier(unsigned *bar, unsigned target, int *err, int *flag) {
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        red_release_add(bar, 1u);
        int good = 1;
        unsigned spins = 0;
        while ((int)(ld_acquire(bar) - target) < 0) {
            if (++spins > kBarrierSpins) {
                atomicOr(err, ERR_BARRIER);
                good = 0;
                break;
            }
            __nanosleep(64);
        }
        if (good && (*(volatile int *)err & ERR_BARRIER)) good = 0;
        *flag = good;
    }
    __syncthreads();
    return *flag != 0;
}

template <int HD, int GP> SYN_DEV void attn_items(const AttnParams &a, int cta, int ncta, float *smem) {
    const int items = a.n_kv * a.splits * a.rows;
    for (int it = cta; it < items; it += ncta) {
        const int g = it % a.n_kv, split = (it / a.n_kv) % a.splits, row = it / (a.n_kv * a.splits);
        attn_compute<HD, GP>(a, g, split, row, smem);
    }
}

// WT: weight type of every GEMV phase; HD, GP: head dimension and padded query-group size of the
// attention phases (one model has one of each, so one kernel holds only the variants it runs).
template <int WT, int HD, int GP>
__global__ void __launch_bounds__(kStepThreads, 1) k_step(const StepParams sp) {
    extern __shared__ __align__(16) float smem[];
    __shared__ float red[32], sv[32];
    __shared__ int si[32], flag, last;
    // The phase descriptor is copied into shared memory: read from global memory, every global
    // store of the phase (outputs, residuals) could alias it and force the compiler to reload
    // pointers and sizes on the critical path of every weight load.
    __shared__ __align__(16) PhaseDesc d;
    const int cta = blockIdx.x, ncta = gridDim.x;
    for (int ph = 0; ph < sp.nphases; ++ph) {
        {
            // every thread must be done with the previous phase's descriptor before it is replaced
            // (the small phases end without a block barrier)
            __syncthreads();
            const int4 *src = reinterpret_cast<const int4 *>(sp.phases + ph);
            int4 *dst = reinterpret_cast<int4 *>(&d);
            for (int i = threadIdx.x; i < (int)(sizeof(PhaseDesc) / 16); i += blockDim.x) dst[i] = __ldg(src + i);
            __syncthreads();
        }
        bool ok = true;
        const bool tr = sp.trace && cta == 0 && threadIdx.x == 0;
        if (tr) sp.trace[3 * ph] = global_ns();
        auto wait = [&] {
            if (ph > 0) ok = grid_barrier(sp.barrier, (unsigned)ph * (unsigned)ncta, sp.err, &flag);
            if (tr) sp.trace[3 * ph + 1] = global_ns();
        };
        switch (d.kind) {
        case PH_GEMV:
            if (d.gemv.gate_up)
                gemv_cta<WT, true, kStepU, kStepThreads / 32>(d.gemv, d.groups, cta, ncta, smem, red, wait);
            else
                gemv_cta<WT, false, kStepU, kStepThreads / 32>(d.gemv, d.groups, cta, ncta, smem, red, wait);
            break;
        case PH_ATTN: {
            const AttnParams &a = d.attn;
            const int items = a.n_kv * a.splits * a.rows;
            for (int it = cta; it < items; it += ncta)
                attn_prefetch(a, it % a.n_kv, (it / a.n_kv) % a.splits, it / (a.n_kv * a.splits));
            wait();
            if (ok) attn_items<HD, GP>(d.attn, cta, ncta, smem);
            break;
        }
        case PH_HEADS:
            wait();
            if (ok) heads_cta(d.heads, cta, ncta);
            break;
        case PH_EMBED:
            wait();
            if (ok) embed_cta(d.embed, cta, ncta);
            break;
        case PH_RMS:
            wait();
            if (ok) rms_cta(d.rms, cta, ncta, red);
            break;
        case PH_ELT:
            wait();
            if (ok) elt_cta(d.elt, cta, ncta);
            break;
        case PH_ARGMAX:
            wait();
            if (ok) argmax_cta(d.argmax, cta, ncta, sv, si, &last);
            break;
        case PH_COPY:
            wait();
            if (ok)
                for (int i = cta * blockDim.x + threadIdx.x; i < d.copy.n; i += ncta * blockDim.x)
                    d.copy.dst[i] = __ldcg(d.copy.src + i);
            break;
        }
        if (tr) sp.trace[3 * ph + 2] = global_ns();
        if (!ok) return;
    }
}

template <int WT, int HD, int GP> int step_blocks_per_sm_t(size_t smem) {
    cudaFuncSetAttribute(k_step<WT, HD, GP>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    int v = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, k_step<WT, HD, GP>, kStepThreads, smem) != cudaSuccess) return 0;
    return v;
}

template <int WT, int HD, int GP> cudaError_t launch_step_t(const StepParams &sp, int blocks, size_t smem, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks);
    cfg.blockDim = dim3(kStepThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeCooperative;
    at[0].val.cooperative = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_step<WT, HD, GP>, sp);
}

// every (head_dim, group) variant of one weight type: a switch over the instantiations
template <int WT> int step_blocks_per_sm_wt(int hd, int gp, size_t smem) {
    switch (hd * 16 + gp) {
    case 64 * 16 + 1: return step_blocks_per_sm_t<WT, 64, 1>(smem);
    case 64 * 16 + 2: return step_blocks_per_sm_t<WT, 64, 2>(smem);
    case 64 * 16 + 4: return step_blocks_per_sm_t<WT, 64, 4>(smem);
    case 64 * 16 + 8: return step_blocks_per_sm_t<WT, 64, 8>(smem);
    case 128 * 16 + 1: return step_blocks_per_sm_t<WT, 128, 1>(smem);
    case 128 * 16 + 2: return step_blocks_per_sm_t<WT, 128, 2>(smem);
    case 128 * 16 + 4: return step_blocks_per_sm_t<WT, 128, 4>(smem);
    case 128 * 16 + 8: return step_blocks_per_sm_t<WT, 128, 8>(smem);
    case 256 * 16 + 1: return step_blocks_per_sm_t<WT, 256, 1>(smem);
    case 256 * 16 + 2: return step_blocks_per_sm_t<WT, 256, 2>(smem);
    case 256 * 16 + 4: return step_blocks_per_sm_t<WT, 256, 4>(smem);
    }
    return 0;
}

template <int WT> cudaError_t launch_step_wt(int hd, int gp, const StepParams &sp, int blocks, size_t smem, cudaStream_t s) {
    switch (hd * 16 + gp) {
    case 64 * 16 + 1: return launch_step_t<WT, 64, 1>(sp, blocks, smem, s);
    case 64 * 16 + 2: return launch_step_t<WT, 64, 2>(sp, blocks, smem, s);
    case 64 * 16 + 4: return launch_step_t<WT, 64, 4>(sp, blocks, smem, s);
    case 64 * 16 + 8: return launch_step_t<WT, 64, 8>(sp, blocks, smem, s);
    case 128 * 16 + 1: return launch_step_t<WT, 128, 1>(sp, blocks, smem, s);
    case 128 * 16 + 2: return launch_step_t<WT, 128, 2>(sp, blocks, smem, s);
    case 128 * 16 + 4: return launch_step_t<WT, 128, 4>(sp, blocks, smem, s);
    case 128 * 16 + 8: return launch_step_t<WT, 128, 8>(sp, blocks, smem, s);
    case 256 * 16 + 1: return launch_step_t<WT, 256, 1>(sp, blocks, smem, s);
    case 256 * 16 + 2: return launch_step_t<WT, 256, 2>(sp, blocks, smem, s);
    case 256 * 16 + 4: return launch_step_t<WT, 256, 4>(sp, blocks, smem, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace syn
