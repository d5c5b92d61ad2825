// tcgen05.cuh -- inline-PTX wrappers for the 5th-generation tensor cores (sm_100 family) as a
// CTA pair uses them: tensor-memory allocation, UMMA issue/commit, TMEM loads and stores, and
// the shared-memory matrix and instruction descriptors for bf16 operands with 128-byte
// swizzle.
#pragma once

#include <stdint.h>

#include "device_common.cuh"

namespace pkv {

// Every tcgen05 instruction of a kernel uses the same CTA group. The kernels here run on CTA
// pairs (a cluster of two CTAs on two SMs): allocation and release are done by one warp of
// each CTA together, and one thread of the pair's leader (cluster rank 0) issues UMMAs that
// read both CTAs' shared memory and write both CTAs' tensor memory.

// ------------------------------------------------------------------ tensor memory
__device__ __forceinline__ void tmem_alloc_pair(uint32_t *dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(dst_smem)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ------------------------------------------------------------------ UMMA (CTA pair)
// D[tmem] (+)= A * B, kind::f16 (bf16 in, fp32 accumulate), M = 256 over the pair: the
// leader's A rows (its shared memory or, in the _ts form, its tensor memory) are rows
// 0..127 and land in its tensor memory, the peer's are rows 128..255 and land in the peer's;
// each CTA holds half of B's N columns at the same shared-memory address (the leader the
// first half). The accumulate flag is an immediate.
template <bool kAccumulate>
__device__ __forceinline__ void umma_pair_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                             uint32_t idesc) {
  if constexpr (kAccumulate)
    asm volatile("tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, 1;" ::"r"(d_tmem),
                 "l"(a_desc), "l"(b_desc), "r"(idesc)
                 : "memory");
  else
    asm volatile("tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, 0;" ::"r"(d_tmem),
                 "l"(a_desc), "l"(b_desc), "r"(idesc)
                 : "memory");
}

// The same with A read from tensor memory (M rows = lanes, each 32-bit column holding two
// consecutive bf16 of K).
template <bool kAccumulate>
__device__ __forceinline__ void umma_pair_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                             uint32_t idesc) {
  if constexpr (kAccumulate)
    asm volatile("tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, 1;" ::"r"(d_tmem),
                 "r"(a_tmem), "l"(b_desc), "r"(idesc)
                 : "memory");
  else
    asm volatile("tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, 0;" ::"r"(d_tmem),
                 "r"(a_tmem), "l"(b_desc), "r"(idesc)
                 : "memory");
}

// Arrive (once) on the mbarrier at shared::cluster address `bar` -- in either CTA of the
// pair -- when every UMMA this thread issued so far has completed.
__device__ __forceinline__ void umma_commit_pair(uint32_t bar_cluster_addr) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          bar_cluster_addr)
      : "memory");
}

// Instruction descriptor, kind::f16: D fp32, A and B bf16, dense, M x N tile.
// a_mn / b_mn select MN-major (1) instead of K-major (0) operand layout.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(uint32_t M, uint32_t N, uint32_t a_mn,
                                                      uint32_t b_mn) {
  return (1u << 4)            // D format: f32
         | (1u << 7)          // A format: bf16
         | (1u << 10)         // B format: bf16
         | (a_mn << 15) | (b_mn << 16) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// Shared-memory matrix descriptor, 128-byte swizzle (tile base 1024-byte aligned).
// lbo / sbo in bytes: for K-major tiles sbo is the stride of 8-row groups (1024) and lbo is
// unused; for MN-major tiles lbo is the stride between 64-element column blocks and sbo the
// stride between 8-row groups along K.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t smem_byte_addr, uint32_t lbo,
                                                    uint32_t sbo) {
  return (uint64_t)((smem_byte_addr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46)  // descriptor version
         | (2ull << 61);                                           // 128-byte swizzle
}

// One lane of the (converged) warp: the lowest active lane. The UMMAs and the commit that
// tracks them have to come from the same thread, which this gives as long as the warp is
// converged at both places.
__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

// ------------------------------------------------------------------ TMEM <-> registers
#define PKV_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), \
                  "=r"(r[i + 4]), "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
#define PKV_W8(i) "r"(r[i]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), "r"(r[i + 4]), \
                  "r"(r[i + 5]), "r"(r[i + 6]), "r"(r[i + 7])
#define PKV_RW8(i) "+r"(r[i]), "+r"(r[i + 1]), "+r"(r[i + 2]), "+r"(r[i + 3]), \
                   "+r"(r[i + 4]), "+r"(r[i + 5]), "+r"(r[i + 6]), "+r"(r[i + 7])

// This warp's 32 TMEM lanes (lane quadrant = warp id % 4, encoded in taddr), 32 consecutive
// 32-bit columns: thread i receives lane (base + i), columns [col, col + 32).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : PKV_R8(0), PKV_R8(8), PKV_R8(16), PKV_R8(24)
      : "r"(taddr));
}

// Wait for this thread's outstanding TMEM loads. The registers pass through the asm so no
// use of them can be scheduled before the wait.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : PKV_RW8(0), PKV_RW8(8), PKV_RW8(16), PKV_RW8(24)
               :
               : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      PKV_W8(0), PKV_W8(8), PKV_W8(16), PKV_W8(24)
      : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      PKV_W8(0), PKV_W8(8)
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Two threads per TMEM lane: 16 consecutive lanes from taddr's lane; threads 0-15 receive
// lane (base + i) at columns [col, col + 32), threads 16-31 lane (base + i - 16) at columns
// [col + kSplit, col + kSplit + 32).
template <int kSplit>
__device__ __forceinline__ void tmem_ld16x2_32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x32bx2.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32], %33;"
      : PKV_R8(0), PKV_R8(8), PKV_R8(16), PKV_R8(24)
      : "r"(taddr), "n"(kSplit));
}

template <int kSplit>
__device__ __forceinline__ void tmem_st16x2_32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x32bx2.x32.b32 [%0], %1, "
      "{%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,"
      "%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33};" ::"r"(taddr),
      "n"(kSplit), PKV_W8(0), PKV_W8(8), PKV_W8(16), PKV_W8(24)
      : "memory");
}

template <int kSplit>
__device__ __forceinline__ void tmem_st16x2_16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x32bx2.x16.b32 [%0], %1, "
      "{%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17};" ::"r"(taddr),
      "n"(kSplit), PKV_W8(0), PKV_W8(8)
      : "memory");
}

#undef PKV_R8
#undef PKV_W8
#undef PKV_RW8

}  // namespace pkv
