// async_dev.cuh -- shared-memory mbarriers and bulk asynchronous copies (TMA), with bounded waits.
// Used by the tensor-core GEMM (k_gemm_tc.cu), the prefill attention on the tensor cores
// (k_attn_tc.cu) and the KV-streaming decode attention (k_attn.cu).
#pragma once

#include <cuda.h>

#include "device_common.cuh"

namespace syn {

constexpr unsigned kAsyncSpin = 1u << 24;   // try_wait polls before a wait gives up

SYN_DEV uint32_t saddr(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

SYN_DEV void mbar_init(uint64_t *b, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(b)), "r"(count) : "memory");
}
// make the initialised barriers visible to the asynchronous proxy (TMA, tensor cores)
SYN_DEV void mbar_init_fence() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

SYN_DEV void mbar_expect_tx(uint64_t *b, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(saddr(b)), "r"(bytes) : "memory");
}
SYN_DEV void mbar_arrive(uint64_t *b) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(saddr(b)) : "memory");
}
SYN_DEV bool mbar_try(uint64_t *b, unsigned parity) {
    unsigned ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(saddr(b)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Non-blocking test of the same phase: true when it has completed.
SYN_DEV bool mbar_test(uint64_t *b, unsigned parity) {
    unsigned ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(saddr(b)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait for the completion of the phase with the given parity. When it runs out, `code` is
// or-ed into *err (if err is set) and false is returned; the caller stops issuing work. A phase that
// has already completed is seen by the non-blocking test, without the potentially blocking form
// (in a clock64 timeline of the prefill attention, the blocking form took a few hundred cycles
// even then).
SYN_DEV bool mbar_wait(uint64_t *b, unsigned parity, int *err, int code) {
    if (mbar_test(b, parity)) return true;
    for (unsigned i = 0; i < kAsyncSpin; ++i)
        if (mbar_try(b, parity)) return true;
    if (err) atomicOr(err, code);
    return false;
}

// Two such waits, whose tests are issued together (one latency when both phases have completed).
SYN_DEV bool mbar_wait2(uint64_t *b1, unsigned p1, uint64_t *b2, unsigned p2, int *err, int code) {
    const bool t1 = mbar_test(b1, p1), t2 = mbar_test(b2, p2);
    if (t1 && t2) return true;
    return (t1 || mbar_wait(b1, p1, err, code)) && (t2 || mbar_wait(b2, p2, err, code));
}

// The same wait with an explicit bound of `spin` polls.
SYN_DEV bool mbar_wait_n(uint64_t *b, unsigned parity, int *err, int code, unsigned spin) {
    if (mbar_test(b, parity)) return true;
    for (unsigned i = 0; i < spin; ++i)
        if (mbar_try(b, parity)) return true;
    if (err) atomicOr(err, code);
    return false;
}

// Contiguous global -> shared copy of `bytes` (multiple of 16; both addresses 16-byte aligned),
// completing on mbarrier `bar` (transaction bytes).
SYN_DEV void bulk_g2s(void *dst, const void *src, unsigned bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     saddr(dst)),
                 "l"(src), "r"(bytes), "r"(saddr(bar))
                 : "memory");
}

// Tiled 2-D tensor copy (TMA) of one box at coordinates (c0 innermost, c1) into shared memory.
SYN_DEV void tma_load_2d(void *dst, const CUtensorMap *map, int c0, int c1, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            saddr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(saddr(bar))
        : "memory");
}

// barrier over the first `threads` threads of the block (named barrier 1), for kernels whose
// producer warp leaves early
SYN_DEV void bar_sync_first(int threads) { asm volatile("bar.sync 1, %0;" ::"r"(threads) : "memory"); }

}  // namespace syn
