// tc_dev.cuh -- 5th-generation tensor-core helpers (tcgen05 MMA, TMEM, descriptors) and the f16
// hi/lo operand split, shared by the bulk-prefill GEMM (k_gemm_tc.cu) and the prefill attention
// (k_attn_tc.cu).
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>

#include "async_dev.cuh"

namespace syn {

// Shared-memory matrix descriptor of a K-major 16-bit tile written with the 128-byte swizzle (by
// TMA, or by threads following the same pattern): rows of 128 bytes, 8-row groups 1024 bytes apart
// (stride byte offset), tile base 1024-aligned; `addr` may step by 32 bytes along K inside a row.
SYN_DEV uint64_t desc_sw128(uint32_t addr) {
    uint64_t d = 0;
    d |= (uint64_t)((addr & 0x3FFFFu) >> 4);      // start address, 16-byte units
    d |= (uint64_t)(16u >> 4) << 16;              // leading byte offset (not used by this layout)
    d |= (uint64_t)(1024u >> 4) << 32;            // stride byte offset: one 8 x 128 B swizzle atom
    d |= (uint64_t)1 << 46;                       // descriptor version of tcgen05
    d |= (uint64_t)2 << 61;                       // swizzle mode: 128-byte
    return d;
}

// The descriptor of an operand `bytes` further on (a multiple of 16): its start address field is the
// shared address / 16 in the low 14 bits, and shared addresses stay below 2^18, so the offset adds
// without a carry out of the field.
SYN_DEV uint32_t desc_off(uint32_t bytes) { return bytes >> 4; }

// Instruction descriptor, kind::f16: f32 accumulator, f16 A and B (format 0), both K-major, M x N.
constexpr uint32_t tc_idesc_f16(int M, int N) {
    return (1u << 4)                              // D format f32
           | ((uint32_t)(N >> 3) << 17)           // N >> 3
           | ((uint32_t)(M >> 4) << 24);          // M >> 4
}

// D (TMEM) = A * B^T (+ D when accumulate != 0); one thread issues it
SYN_DEV void mma_f16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(tmem_d),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}
// arrive on `bar` once every tcgen05 operation this thread issued so far has completed
SYN_DEV void mma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(saddr(bar))
                 : "memory");
}
SYN_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
SYN_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// one warp: allocate / free `cols` TMEM columns (a power of two >= 32); the base address is
// written to shared memory
SYN_DEV void tmem_alloc(uint32_t *dst, uint32_t cols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(dst)), "r"(cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
SYN_DEV void tmem_free(uint32_t base, uint32_t cols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(base), "r"(cols) : "memory");
}

// 32 lanes x 32 consecutive f32 columns: thread t of the warp gets lane (base lane + t)
SYN_DEV void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// the same load without its wait: several loads may be in flight before one tmem_ld_wait()
SYN_DEV void tmem_ld32_issue(uint32_t taddr, uint32_t *r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
// 32 lanes x 16 consecutive f32 columns, without the wait
SYN_DEV void tmem_ld16_issue(uint32_t taddr, uint32_t *r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
// wait for this thread's TMEM loads; their registers may be read only after it
SYN_DEV void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// make this thread's generic shared-memory stores visible to the tensor core (async proxy)
SYN_DEV void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// power of two that brings a vector whose largest magnitude is amax just under 2^14 (inside the f16
// range, with headroom); 1 for zero or non-finite input
SYN_DEV float row_scale(float amax) {
    if (!(amax > 0.f) || !isfinite(amax)) return 1.f;
    int e;
    frexpf(amax, &e);   // amax < 2^e
    return ldexpf(1.f, 14 - e);
}

// v = h + l with h = f16(v), l = f16(v - h): 22 significant bits in two halves
SYN_DEV void split2(float v, __half &h, __half &l) {
    h = __float2half_rn(v);
    l = __float2half_rn(v - __half2float(h));
}

// Host: tensor map of a row-major [rows][cols] f16 plane (cols * 2 bytes a multiple of 16, base
// 16-byte aligned) for TMA loads of 64-column x box_rows boxes with the 128-byte swizzle; elements
// outside the plane read as zero. False when the driver entry point is unavailable or the encoder
// rejects the layout. Defined in k_gemm_tc.cu.
bool tma_map_f16(CUtensorMap *map, const void *base, int64_t rows, int64_t cols, int box_rows);
// Host: whether the driver's tensor-map encoder could be reached (defined in k_gemm_tc.cu).
bool tma_encoder_available();

}  // namespace syn
