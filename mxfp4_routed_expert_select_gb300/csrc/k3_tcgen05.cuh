// k3_tcgen05.cuh -- small helpers for tcgen05 / TMA kernels (sm_103a):
// shared-memory matrix descriptors, MMA commits, tcgen05 fences, tiled TMA
// loads, TMEM loads and bounded barrier waits.
#pragma once
#include <cuda.h>
#include <cudaTypedefs.h>

#include "k3_device.cuh"

namespace k3 {

K3_DEV uint32_t smem_addr(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

// Shared-memory matrix descriptor of a K-major operand with the 128-byte
// swizzle, split in its two 32-bit halves.  Low half: start address >> 4
// (bits 0-13) and leading byte offset 1 (bits 16-29, unused with this
// swizzle); it is the only half that changes, and +32 bytes of K is +2.
// High half: stride byte offset 1024 >> 4 (8-row groups 1024 bytes apart),
// descriptor version 1 (bit 46 of the whole), swizzle mode 2 (bits 61-63).
K3_DEV uint32_t sw128_lo(uint32_t saddr) { return ((saddr & 0x3FFFFu) >> 4) | (1u << 16); }
constexpr uint32_t SW128_HI = (1024u >> 4) | (1u << 14) | (2u << 29);
// Commit by the lane elect.sync picks (the lane that issued the MMAs).
K3_DEV void mma_commit(uint32_t bar)
{
    asm volatile("{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
                 "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
                 : "memory");
}
K3_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
K3_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
K3_DEV void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// 2D tiled TMA load (x = byte column, a multiple of 16; y = row).
K3_DEV void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar)
{
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
                 "%3}], [%4];" ::"r"(dst),
                 "l"((uint64_t)map), "r"(x), "r"(y), "r"(bar)
                 : "memory");
}

// L2 policy for data a launch reads once (the expert weights and router
// rows): evicted first, so that streaming them does not push out of L2 what
// the launch reuses -- its own instructions, the activation and h images,
// partial sums and counters -- which would otherwise come back from HBM at
// every first use.
K3_DEV uint64_t l2_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
// tma_load_2d with an L2 cache policy.
K3_DEV void tma_load_2d_hint(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar, uint64_t policy)
{
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
                 "[%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
                 "l"((uint64_t)map), "r"(x), "r"(y), "r"(bar), "l"(policy)
                 : "memory");
}
// bulk_g2s with an L2 cache policy.
K3_DEV void bulk_g2s_hint(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar, uint64_t policy)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, "
                 "[%3], %4;" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar), "l"(policy)
                 : "memory");
}

// A hint: bring one TMA tile (x = byte column, y = row) of `map` into L2.
// Nothing waits for it; a later load of the same tile hits L2 if the line is
// still there.
K3_DEV void tma_prefetch_l2_2d(const CUtensorMap *map, int x, int y)
{
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"((uint64_t)map), "r"(x),
                 "r"(y)
                 : "memory");
}

// 8 consecutive fp32 columns (column address a multiple of 8).
K3_DEV void tmem_ld8(uint32_t taddr, float (&v)[8])
{
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                   "=r"(r[7])
                 : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 8; i++) v[i] = __uint_as_float(r[i]);
}
K3_DEV void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

K3_DEV bool tc_wait(uint32_t bar, uint32_t parity, int *err, volatile int *abort_flag)
{
    if (*abort_flag) return false;
    if (!mbar_wait(bar, parity, err)) {
        *abort_flag = 1;
        return false;
    }
    return true;
}


}  // namespace k3
