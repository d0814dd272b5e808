// tcgen05 (5th-generation tensor core) helpers: TMEM allocation, MMA issue and commit,
// TMEM loads, and shared-memory matrix descriptors for the 128-byte-swizzled K-major
// canonical layout (PTX ISA, "tcgen05" sections: instruction descriptor, matrix
// descriptor, data movement shapes).
#pragma once

#include "tma.cuh"

namespace fq {

// ---- tensor memory (one warp, .sync.aligned)
FQ_DEV void tmem_alloc(uint32_t* smem_dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_dst)),
                 "r"(ncols)
                 : "memory");
}
FQ_DEV void tmem_relinquish() { asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory"); }
FQ_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
FQ_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
FQ_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// generic-proxy shared-memory writes -> visible to the async proxy (tensor core reads)
FQ_DEV void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// ---- MMA: D[tmem] (+)= A[smem] x B[smem], kind::f16, one thread issues
FQ_DEV void mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// arrive once on bar when every MMA issued so far by this thread has completed
FQ_DEV void mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// Instruction descriptor, kind::f16: D f32, A and B f16, both K-major, shape M x N.
//   bits 4-5 D format (1 = f32); 7-9 A format (0 = f16); 10-12 B format (0 = f16);
//   15 / 16 A / B major (0 = K); 17-22 N >> 3; 24-28 M >> 4.
FQ_HD constexpr uint32_t idesc_f16_f32(int M, int N) {
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Shared-memory matrix descriptor for a K-major operand in the 128-byte swizzled canonical
// layout: 8-row x 128-byte atoms stacked along M/N every 1024 bytes (stride byte offset),
// the 16-byte chunk index of each row XORed with the row index within the atom.
//   bits 0-13 start address >> 4; 16-29 leading byte offset >> 4 (unused here, 1);
//   32-45 stride byte offset >> 4; 46-47 version (1); 61-63 layout (2 = 128-byte swizzle).
FQ_DEV uint64_t sdesc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// byte offset of (row, 16-byte chunk j of its 128-byte K slice) in the swizzled layout
FQ_DEV uint32_t sw128_offset(int row, int j) {
    return (uint32_t)((row >> 3) * 1024 + (row & 7) * 128 + ((j ^ (row & 7)) << 4));
}

// ---- TMEM -> registers: 32 lanes x 32 bits, 16 consecutive columns per thread
FQ_DEV void tmem_ld16(uint32_t taddr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}
FQ_DEV void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

}  // namespace fq
