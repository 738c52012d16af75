// Fifth-generation tensor-core (tcgen05) and tensor-memory-access (TMA)
// wrappers for sm_103a, as inline PTX: tensor-memory allocation, loads and
// stores (registers <-> tensor memory), the CTA-pair bf16 x bf16 -> FP32 MMA
// with operands in shared memory and its commit to the pair's mbarriers, 2-D
// tiled TMA loads, and the two 32/64-bit descriptors the MMA takes.
#pragma once
#include <cuda.h>

#include "rbi_device.cuh"

namespace rbi {
namespace umma {

// ---------------------------------------------------------------- tensor memory

// Allocates `ncols` columns (a power of two >= 32) of this CTA's tensor memory
// and writes the base address to *slot (shared memory).  One whole warp.
__device__ __forceinline__ void tmem_alloc(uint32_t *slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(slot)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
// One whole warp (the one that allocated).
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Ordering of tcgen05 operations across a thread synchronisation (barrier,
// mbarrier wait): `before` ahead of the sync in the thread that issued them,
// `after` behind the sync in the thread that continues.
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive FP32 columns of the warp's 32 lanes: lane l gets tensor-memory
// lane (taddr.lane + l), columns taddr.col .. +31.  Whole warp; the values are
// valid after wait_ld().
__device__ __forceinline__ void ld_32x32(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
          "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
          "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 8 consecutive 32-bit columns of the warp's 32 lanes, registers -> tensor
// memory and back (lane l: tensor-memory lane taddr.lane + l).  Whole warp;
// the stores are complete after wait_st(), the loaded values valid after
// wait_ld().
__device__ __forceinline__ void st_32x32_x8(uint32_t taddr, const uint32_t (&v)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(v[0]),
                 "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                 : "memory");
}
__device__ __forceinline__ void ld_32x32_x8(uint32_t taddr, uint32_t (&v)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
                 : "r"(taddr)
                 : "memory");
}
__device__ __forceinline__ void wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ---------------------------------------------------------------- CTA pairs (cta_group::2)
//
// A pair of CTAs (ranks 0 and 1 of a 2-CTA cluster, on two SMs) runs one MMA
// of twice the rows: each CTA holds half of A (its M/2 rows) and half of B
// (its N/2 columns) in its own shared memory at the same offsets, the MMA is
// issued by one thread of rank 0, and each CTA's tensor memory receives its
// M/2 rows of D (all N columns).  Allocation and release of tensor memory are
// performed by one warp of each CTA of the pair.

__device__ __forceinline__ void tmem_alloc_pair(uint32_t *slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(slot)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void mma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                              uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// One arrival on the mbarrier at this offset in every CTA of `cta_mask` once
// the pair MMAs this thread issued so far have completed.
__device__ __forceinline__ void commit_pair_multicast(uint64_t *bar, uint16_t cta_mask) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_addr(bar)),
        "h"(cta_mask)
        : "memory");
}

// ---------------------------------------------------------------- TMA

// Box of a 2-D tiled tensor map at element coordinates (x inner, y outer) into
// this CTA's shared memory; completion counted in bytes on `bar`.  x times the
// element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int32_t x, int32_t y,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

// The same load issued by rank 1 of a CTA pair into its own shared memory,
// with completion counted on an mbarrier of rank 0 (`bar_cluster`: a
// shared::cluster address of the peer's barrier).
__device__ __forceinline__ void tma_load_2d_to_peer_bar(void *dst, const CUtensorMap *map, int32_t x, int32_t y,
                                                        uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2 [%0], [%1, "
        "{%2, %3}], [%4];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cluster)
        : "memory");
}

// ---------------------------------------------------------------- descriptors

// Shared-memory matrix descriptor of an operand tile in the canonical
// MN-major layout with the 128-byte swizzle: rows of 64 bf16 along M (or N)
// at one k, 128 bytes each, eight k-rows per 1024-byte swizzle atom.
//   bits  0-13  start address >> 4
//   bits 16-29  leading byte offset >> 4: from one 64-element M/N chunk to the next
//   bits 32-45  stride byte offset >> 4: from one group of eight k-rows to the next
//   bits 46-47  descriptor version (1)
//   bits 61-63  layout: 2 = 128-byte swizzle
// The tile must start on a 1024-byte boundary (base offset 0).
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
    return uint64_t((saddr >> 4) & 0x3fffu) | (uint64_t((lbo_bytes >> 4) & 0x3fffu) << 16) |
           (uint64_t((sbo_bytes >> 4) & 0x3fffu) << 32) | (uint64_t(1) << 46) | (uint64_t(2) << 61);
}

// Instruction descriptor of kind::f16 with bf16 A and B, FP32 D, both
// operands MN-major, shape M x N (x K = 16):
//   bits 4-5 D format (1 = F32), 7-9 A format (1 = BF16), 10-12 B format
//   (1 = BF16), 15 A major (1 = MN), 16 B major (1 = MN), 17-22 N >> 3,
//   24-28 M >> 4.
__host__ __device__ constexpr uint32_t idesc_bf16_mn(uint32_t M, uint32_t N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | (1u << 15) | (1u << 16) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

}  // namespace umma
}  // namespace rbi
