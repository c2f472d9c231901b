// Fifth-generation tensor core (tcgen05) helpers for sm_103a, inline PTX:
// shared-memory matrix descriptors, the bf16 instruction descriptor, MMA
// issue and commit, tensor-memory allocation and loads, mbarriers and TMA.
//
// Operand layouts used with these helpers (all 128-byte swizzled, tiles
// 1024-byte aligned, as a TMA copy with CU_TENSOR_MAP_SWIZZLE_128B writes
// them):
//   K-major  rows of 64 bf16 (128 B) along K; 8-row groups 1024 B apart
//            (stride byte offset 1024); a K extent of 128 is two such
//            chunks; one K=16 step advances the start address by 32 B.
//   MN-major rows of 64 bf16 along M or N, one row per K index; 8-row groups
//            1024 B apart (stride byte offset), 64-wide chunks along M or N
//            `chunk` bytes apart (leading byte offset); one K=16 step
//            advances the start address by 16 rows (2048 B).
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace mita {
namespace tc {

MITA_DEV uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

// Shared-memory matrix descriptor (128-byte swizzle).
MITA_DEV uint64_t desc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;   // descriptor version
    d |= (uint64_t)2 << 61;   // 128-byte swizzle
    return d;
}
MITA_DEV uint64_t desc_kmajor(uint32_t saddr) { return desc_sw128(saddr, 16u, 1024u); }
MITA_DEV uint64_t desc_mnmajor(uint32_t saddr, uint32_t chunk_bytes) { return desc_sw128(saddr, chunk_bytes, 1024u); }

// Instruction descriptor: bf16 x bf16 -> fp32, M x N, operand majors
// (0 = K-major, 1 = M/N-major).
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int a_mn, int b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= A . B^T, issued by one thread.
MITA_DEV void mma_bf16(uint32_t tmem_d, uint64_t da, uint64_t db, uint32_t idesc, bool accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.u32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(
            tmem_d),
        "l"(da), "l"(db), "r"(idesc), "r"((uint32_t)accumulate));
}
// The mbarrier receives one arrival when every MMA this thread issued so far is done.
MITA_DEV void mma_commit(uint32_t mbar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(mbar)
                 : "memory");
}
MITA_DEV void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }
MITA_DEV void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }

// Tensor memory: one warp allocates / frees `cols` columns (a power of two >= 32).
MITA_DEV void tmem_alloc(uint32_t slot_saddr, uint32_t cols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(slot_saddr), "r"(cols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
}
MITA_DEV void tmem_free(uint32_t taddr, uint32_t cols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(cols));
}
// 32 consecutive fp32 columns of this thread's lane (the warp reads lanes 32 (warp % 4) + lane).
MITA_DEV void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
        "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}

// ---------------------------------------------------------------- mbarrier / TMA
MITA_DEV void mbar_init(uint32_t bar, int count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count));
}
MITA_DEV void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory"); }
MITA_DEV void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes) : "memory");
}
MITA_DEV bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Wait for the phase with the given parity, giving up after `budget` SM
// cycles (about a second by default; returns false and the caller reports
// MITA_ERR_TIMEOUT).
MITA_DEV bool mbar_wait_bounded(uint32_t bar, uint32_t parity, long long budget = 2000000000LL) {
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity))
        if (clock64() - t0 > budget) return false;
    return true;
}
MITA_DEV void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];\n" ::"r"(dst),
        "l"(map), "r"(x), "r"(y), "r"(bar)
        : "memory");
}
MITA_DEV void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }

}  // namespace tc
}  // namespace mita
