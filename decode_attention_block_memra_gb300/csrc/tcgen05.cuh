// Fifth-generation tensor cores (tcgen05) from inline PTX: tensor-memory
// allocation, single-thread MMA issue with both operands in shared memory and
// the fp32 accumulator in tensor memory, completion through an mbarrier, and
// tensor-memory loads into registers.
//
// Operands use the no-swizzle K-major canonical layout: the matrix is cut into
// core matrices of 8 rows x 16 bytes (8 fp16 along K), each stored as 128
// contiguous bytes (row i of the core matrix at byte 16 i).  Our tiles place
// core matrix (row group g, K group k) at ((g * K/8) + k) * 128, so the two
// core matrices one K = 16 step reads are 128 bytes apart (the leading
// byte offset) and row groups are K/8 * 128 bytes apart (the stride byte
// offset); the next K step starts 256 bytes further on.
#pragma once

#include <stdint.h>

namespace memra {
namespace tc {

// Matrix descriptor of a no-swizzle operand in shared memory: start address,
// leading byte offset (between the core matrices adjacent along K), stride
// byte offset (between core matrices adjacent along M or N), the fixed
// descriptor version 1 at bit 46; base offset 0, swizzle mode 0.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((addr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}

// Instruction descriptor of an MMA of kind::f16: fp32 accumulator (bits 4-5 =
// 1), A and B fp16 (bits 7-9, 10-12 = 0), neither negated, both K-major (bits
// 15, 16 = 0), N / 8 at bits 17-22, M / 16 at bits 24-28.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {
  return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// Whole warp: allocate `ncols` tensor-memory columns (a power of two, 32 ..
// 512); the base address is written to the shared-memory word at `slot`.
__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot), "r"(ncols)
               : "memory");
}

// Whole warp: this CTA will allocate no more tensor memory.
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

// Whole warp: free what tmem_alloc returned.
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Order tcgen05 operations around a thread barrier.
__device__ __forceinline__ void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// One thread: D[tmem] (+)= A[smem] * B[smem]^T, M x N x 16, fp16 in, fp32
// accumulate; accumulate = 0 overwrites D.
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// One thread: arrive once on the mbarrier when every MMA this thread issued
// before has completed (its shared-memory reads included).
__device__ __forceinline__ void commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// Whole warp: lane i of the warp reads tensor-memory lane (lane field of
// `taddr`) + i, 16 consecutive 32-bit columns from the column of `taddr`.  A
// warp may only address the 32 lanes of its own quarter (warp id % 4).  The
// registers are valid after wait_ld, which takes them as operands so that no
// use can move above it.
__device__ __forceinline__ void ld_32x32b_x16(uint32_t taddr, uint32_t *r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

__device__ __forceinline__ void wait_ld(uint32_t *r) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15])
               :
               : "memory");
}

// Whole warp: the store counterpart of ld_32x32b_x16 (lane i of the warp
// writes its 16 registers to tensor-memory lane (lane field of `taddr`) + i).
__device__ __forceinline__ void st_32x32b_x16(uint32_t taddr, const uint32_t *r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

// Whole warp: this thread's earlier tensor-memory stores have completed.
__device__ __forceinline__ void wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

}  // namespace tc
}  // namespace memra
