// Bulk asynchronous copies (TMA, 1-D) and mbarriers for staging weight chunks into shared
// memory.  Every wait is bounded by a clock budget so that a kernel can report a stuck
// pipeline through an error word instead of spinning forever.
#pragma once

#include "common.cuh"

namespace fq {

FQ_DEV uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

FQ_DEV void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
FQ_DEV void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

FQ_DEV void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
FQ_DEV void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
FQ_DEV bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// About a quarter second at GB300 clocks: far beyond any legitimate wait inside one kernel.
constexpr long long WAIT_BUDGET_CYCLES = 1ll << 29;

// Wait for the phase with the given parity to complete; false once the budget is spent.
FQ_DEV bool mbar_wait(uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > WAIT_BUDGET_CYCLES) return false;
    return true;
}

// dst (shared, 16-byte aligned) <- src (global, 16-byte aligned), bytes a multiple of 16;
// completion is counted on bar's transaction count.
FQ_DEV void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// 2-D tiled copy of the box at (x, y) of the tensor described by tmap (a __grid_constant__
// kernel parameter) into shared memory (128-byte aligned); x * element size must be a
// multiple of 16 bytes.  Out-of-range parts of the box are zero-filled and still counted.
FQ_DEV void tma_load_2d(void* dst, const void* tmap, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(dst)),
        "l"(tmap), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// Named barrier over the first `threads` threads of the CTA (id 1; id 0 is __syncthreads).
FQ_DEV void bar_sync_consumers(int threads) { asm volatile("bar.sync 1, %0;" ::"r"(threads) : "memory"); }

}  // namespace fq
