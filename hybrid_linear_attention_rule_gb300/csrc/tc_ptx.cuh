// tc_ptx.cuh -- thin inline-PTX wrappers for the sm_100-family tensor-core path
// (tcgen05 MMA with TMEM accumulators, shared-memory matrix descriptors,
// mbarriers).  Written from the public PTX ISA description of these
// instructions; every wait is bounded by the caller.
#pragma once

#include <stdint.h>

namespace k3kda {
namespace tc {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// The dynamic shared-memory window rounded up to a 1024-byte boundary, derived from the shared
// array by pointer arithmetic so that the compiler still knows every access through it to be a
// shared one (a round trip through an integer would leave it a generic pointer).
__device__ __forceinline__ uint8_t *smem_align1024(uint8_t *base) {
    return base + ((1024u - (smem_u32(base) & 1023u)) & 1023u);
}

// ---- mbarrier ----
__device__ __forceinline__ void mbar_init(uint32_t addr, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(addr), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t addr, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(addr), "r"(parity)
        : "memory");
    return ok != 0;
}
// Spin until the phase with the given parity completes; false after max_iters tries.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t addr, uint32_t parity, uint32_t max_iters) {
    for (uint32_t i = 0; i < max_iters; ++i)
        if (mbar_try_wait(addr, parity)) return true;
    return false;
}

// ---- fences ----
__device__ __forceinline__ void fence_async_smem() {   // generic-proxy smem writes -> visible to tcgen05
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// ---- tensor memory allocation (one full warp) ----
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// ---- descriptors ----
// K-major operand tile with the 128-byte swizzle: rows of 64 bf16 (128 B), 8-row
// groups of 1024 B, tile base 1024-byte aligned.  Advancing K by 16 elements
// inside the 64-element row is a +32 B start address.
__device__ __forceinline__ uint64_t sdesc_kmajor_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);       // start address (16 B units)
    d |= (uint64_t)1 << 16;                           // leading byte offset (unused for this layout)
    d |= (uint64_t)(1024u >> 4) << 32;                // stride byte offset: 8-row group pitch
    d |= (uint64_t)1 << 46;                           // descriptor version for tcgen05
    d |= (uint64_t)2 << 61;                           // swizzle mode: 128 B
    return d;
}

// MN-major operand tile with the 128-byte swizzle: K rows of 64 contiguous MN
// elements (128 B), 8-row K groups of 1024 B; successive 64-element MN blocks
// lie mn_block_bytes apart.  Advancing K by 16 rows is a +2048 B start address.
__device__ __forceinline__ uint64_t sdesc_mnmajor_sw128(uint32_t saddr, uint32_t mn_block_bytes) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);             // start address (16 B units)
    d |= (uint64_t)((mn_block_bytes >> 4) & 0x3FFFu) << 16; // leading byte offset: MN block pitch
    d |= (uint64_t)(1024u >> 4) << 32;                      // stride byte offset: 8-row K group pitch
    d |= (uint64_t)1 << 46;                                 // descriptor version for tcgen05
    d |= (uint64_t)2 << 61;                                 // swizzle mode: 128 B
    return d;
}

// Advance a shared-memory descriptor's start address by `bytes` (a multiple of 16, no carry
// out of the 14-bit field for addresses below 256 KB).
__device__ __forceinline__ uint64_t dadd(uint64_t desc, uint32_t bytes) { return desc + (bytes >> 4); }

// Instruction descriptor, kind::f16 with bf16 A and B, fp32 accumulator, both K-major
// unless a_mn / b_mn select the MN-major layout for that operand.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool negate_a = false, bool a_mn = false,
                                                      bool b_mn = false) {
    return (1u << 4)                                  // D format: f32
           | (1u << 7)                                // A format: bf16
           | (1u << 10)                               // B format: bf16
           | ((negate_a ? 1u : 0u) << 13)             // negate A
           | ((a_mn ? 1u : 0u) << 15)                 // A major: MN
           | ((b_mn ? 1u : 0u) << 16)                 // B major: MN
           | ((uint32_t)(N >> 3) << 17)               // N / 8
           | ((uint32_t)(M >> 4) << 24);              // M / 16
}

// Instruction descriptor, kind::tf32 (A and B fp32 words read as tf32), fp32 accumulator, both
// operands K-major.
__host__ __device__ constexpr uint32_t idesc_tf32_f32(int M, int N) {
    return (1u << 4)                                  // D format: f32
           | (2u << 7)                                // A format: tf32
           | (2u << 10)                               // B format: tf32
           | ((uint32_t)(N >> 3) << 17)               // N / 8
           | ((uint32_t)(M >> 4) << 24);              // M / 16
}

// ---- MMA issue (single thread) and completion ----
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Same MMA with the A operand (M rows x 16 K, bf16 pairs packed per 32-bit column, K-major)
// read from tensor memory at a_tmem instead of shared memory.
__device__ __forceinline__ void mma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
        ::"r"(d_tmem), "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// kind::tf32 MMA, both operands in shared memory (descriptors).
__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// kind::tf32 MMA with A (M rows x 8 K, one fp32 word per column) read from tensor memory.
__device__ __forceinline__ void mma_tf32_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}"
        ::"r"(d_tmem), "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t mbar_smem) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar_smem)
                 : "memory");
}

// ---- TMEM <-> registers (a warp accesses the 32 lanes of its sub-partition) ----
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
        ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
          "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
        ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
        : "memory");
}
__device__ __forceinline__ void tmem_ld4(uint32_t taddr, uint32_t (&r)[4]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(taddr));
}
__device__ __forceinline__ void tmem_st4(uint32_t taddr, const uint32_t (&r)[4]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};"
                 ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3])
                 : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// x = hi + lo with hi rounded to the nearest tf32 value (low 13 mantissa bits zero) and lo the
// exact fp32 remainder: a kind::tf32 product hi.hi + hi.lo + lo.hi then carries about 21 bits.
__device__ __forceinline__ void split_tf32(float x, uint32_t &hi, uint32_t &lo) {
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(hi) : "f"(x));
    lo = __float_as_uint(x - __uint_as_float(hi));
}
// Byte offset of fp32 element (row, k) in a K-major 128B-swizzled tile: 32 elements of K per
// 128-byte row, 8-row groups of 1024 B, successive 32-element K atoms atom_bytes apart.
__device__ __forceinline__ uint32_t sw128_offset_f32(uint32_t row, uint32_t k, uint32_t atom_bytes) {
    const uint32_t byte = (k & 31u) * 4u;
    return (k >> 5) * atom_bytes + (row >> 3) * 1024u + (row & 7u) * 128u +
           ((((byte >> 4) ^ (row & 7u)) << 4) | (byte & 15u));
}
// Byte offset of element (row, col) in a K-major 128B-swizzled bf16 tile whose
// rows hold 64 elements (one swizzle atom wide); col < 64.
__device__ __forceinline__ uint32_t sw128_offset(uint32_t row, uint32_t col) {
    const uint32_t byte = col * 2u;
    return (row >> 3) * 1024u + (row & 7u) * 128u + ((((byte >> 4) ^ (row & 7u)) << 4) | (byte & 15u));
}

}  // namespace tc
}  // namespace k3kda

namespace k3kda {
namespace tc {

// ---- bulk (non-tensor) async copies global -> shared, completing on an mbarrier ----
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t mbar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(mbar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t mbar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(mbar) : "memory");
}
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst_smem, const void *src, uint32_t bytes, uint32_t mbar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst_smem), "l"(src), "r"(bytes), "r"(mbar)
                 : "memory");
}
// Tiled TMA load of a 3-D box (coordinates innermost first) into shared memory,
// completing on an mbarrier.  tmap is the generic address of a CUtensorMap held in
// kernel-parameter (grid-constant) memory.
__device__ __forceinline__ void tma_load_3d(uint32_t dst_smem, const void *tmap, int x, int y, int z, uint32_t mbar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
        ::"r"(dst_smem), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(mbar)
        : "memory");
}
// Bulk copy shared -> global in the issuing thread's bulk-async group (both addresses
// 16-byte aligned, bytes a multiple of 16).  Sources must have been made visible to
// the async proxy (fence.proxy.async) by their writers first.
__device__ __forceinline__ void bulk_s2g(void *dst, uint32_t src_smem, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                 ::"l"(dst), "r"(src_smem), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Prefetch [src, src + bytes) from global memory into L2 (src 16-byte aligned, bytes a multiple
// of 16); nothing signals completion, a later copy of the same bytes just finds them in L2.
__device__ __forceinline__ void prefetch_l2(const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
// Prefetch the 3-D map's box at {x, y, z} into L2.
__device__ __forceinline__ void tma_prefetch_3d(const void *tmap, int x, int y, int z) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];"
                 ::"l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z)
                 : "memory");
}
// TMA tensor store shared -> global of the 3-D map's box at {x, y, z}, in the issuing thread's
// bulk-async group; box rows outside the tensor are not written.  The writers of the source
// must have fenced it to the async proxy (fence.proxy.async) first.
__device__ __forceinline__ void tma_store_3d(const void *tmap, uint32_t src_smem, int x, int y, int z) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];"
                 ::"l"(reinterpret_cast<uint64_t>(tmap)), "r"(src_smem), "r"(x), "r"(y), "r"(z)
                 : "memory");
}
// Wait until every committed bulk group of this thread has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Same, except that the most recently committed group may still be reading.
__device__ __forceinline__ void bulk_wait_read_but_last() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
// Wait until every committed bulk group of this thread has completed (writes performed).
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Named barrier over `count` threads (a multiple of 32).
__device__ __forceinline__ void named_bar(uint32_t id, uint32_t count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

}  // namespace tc
}  // namespace k3kda
