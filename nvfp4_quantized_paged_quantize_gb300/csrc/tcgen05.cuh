// tcgen05.cuh -- fifth-generation tensor-core building blocks for sm_103a,
// written as inline PTX: tensor-memory (TMEM) allocation, shared-memory matrix
// descriptors, the instruction descriptor of kind::f16, the single-thread MMA
// issue with its mbarrier commit, and the warp-wide TMEM loads and stores.
//
// Everything here is the CTA-pair form (.cta_group::2): two CTAs of a
// cluster, ranks 0 and 1, on two SMs.  Each allocates the same TMEM columns;
// one thread of rank 0 issues an MMA of M = 256 whose rows 0-127 live in rank
// 0's TMEM and rows 128-255 in rank 1's (A read from TMEM, D written to it),
// while the shared-memory B operand is split by N: each CTA holds half of its
// columns at the same shared-memory address.  Every tcgen05 instruction of a
// kernel uses the same CTA-group form.
//
// Operand layouts in shared memory are the no-swizzle canonical ones: a "core
// matrix" is 8 rows of 16 bytes stored as 128 contiguous bytes.
//  - K-major operand (rows = M or N, K contiguous within a row): core matrix
//    (row group i, K chunk j) at i * SBO + j * LBO; inside it, row r at r * 16.
//  - MN-major operand (K rows, M or N contiguous within a row): core matrix
//    (MN group i, K group j) at i * SBO + j * LBO; inside it, K row r at r * 16.
// One kind::f16 MMA consumes K = 16, i.e. two core matrices along K.
#pragma once

#include <cstdint>

namespace nvfp4kv {
namespace tc {

// Allocate ncols (a power of two >= 32) TMEM columns in both CTAs of the
// pair; the TMEM address is written to shared memory at dst.  Executed by one
// whole warp in each of the two CTAs.
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

// Free the allocation (the allocating warps, after every TMEM access of the pair).
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Order tcgen05 operations against thread synchronisation (barriers, mbarrier
// waits): "before" ahead of the sync, "after" behind it.
__device__ __forceinline__ void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Make this thread's ordinary shared-memory stores visible to the tensor core
// (the asynchronous proxy); placed before the barrier that publishes them.
__device__ __forceinline__ void fence_smem_to_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Shared-memory matrix descriptor: start address, leading-dimension byte
// offset (LBO), stride-dimension byte offset (SBO), all in 16-byte units;
// bits 46-47 hold the descriptor version (1), the layout field (bits 61-63)
// stays 0: no swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}

// Instruction descriptor of kind::f16 with f16 A and B and an f32 accumulator:
// bits 4-5 accumulator format (1 = f32), 7-9 / 10-12 A / B format (0 = f16),
// 15 / 16 A / B major-ness (1 = MN-major), 17-22 N / 8, 24-28 M / 16.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int m, int n, bool a_mn_major, bool b_mn_major) {
  return (1u << 4) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
         ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// D (TMEM) = A * B (+ D when accumulate != 0) over the pair, with A read from
// TMEM: in each CTA lane r holds its row r, each 32-bit column two consecutive
// K elements (the lower K index in the low half); one kind::f16 MMA reads 8
// columns (K = 16).  Issued by one thread of rank 0.
__device__ __forceinline__ void mma_f16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                               uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on the issuing CTA's mbarrier when every MMA this thread issued
// so far is done.
__device__ __forceinline__ void commit(uint32_t mbar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar)
               : "memory");
}

// The same, arriving on the mbarrier at this shared-memory offset in each CTA
// of cta_mask (bit k: cluster rank k).
__device__ __forceinline__ void commit_multicast(uint32_t mbar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(mbar),
      "h"(cta_mask)
      : "memory");
}

// Warp-wide TMEM load: thread i gets lane (lane field of taddr) + i, 32
// consecutive 32-bit columns from the column of taddr.  The wait is part of
// the same statement, so no use of r can be scheduled before the data lands.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

// Warp-wide TMEM store of the same shape; waits for completion.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

}  // namespace tc
}  // namespace nvfp4kv
