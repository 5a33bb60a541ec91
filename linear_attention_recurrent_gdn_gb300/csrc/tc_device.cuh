// 5th-generation tensor-core building blocks (sm_100a / sm_103a) in inline PTX:
// tensor-memory (TMEM) allocation, tcgen05.mma with bf16 operands and fp32
// accumulation, its completion on an mbarrier, and TMEM loads.
//
// Operand layout used throughout: K-major with no swizzle.  A matrix of R rows
// and K columns of bf16 is stored as 8-row x 16-byte "core matrices" (128
// contiguous bytes, row r of the core matrix at byte 16 * r); core matrix
// (r / 8, k / 8) sits at byte ((r / 8) * (K / 8) + k / 8) * 128.  In the shared
// memory descriptor the leading-dimension offset (between core matrices
// adjacent along K) is then 128 bytes and the stride-dimension offset (between
// adjacent 8-row groups) is K / 8 * 128 bytes; one MMA of K = 16 reads two core
// matrices along K, so the next K step starts 256 bytes further.
//
// The accumulator of an M = 128 MMA holds row m in TMEM lane m and column n in
// TMEM column (base + n); warp w of a CTA may read lanes 32 * (w % 4) .. +31.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace dl {
namespace tc {

// Byte offset of element (r, k) in a K-major, no-swizzle bf16 operand with K columns.
__host__ __device__ constexpr uint32_t kmaj_off(int r, int k, int K) {
  return (uint32_t)((((r >> 3) * (K >> 3)) + (k >> 3)) * 128 + (r & 7) * 16 + (k & 7) * 2);
}
// The same operand stored MN-major, no swizzle: the core matrix at the same
// place holds eight K indices as 16-byte rows, each with eight consecutive
// rows r of the operand, so a K index's eight values of r are one 16-byte
// store.  The shared-memory descriptor is the same as for kmaj_off (leading
// offset 128 bytes between core matrices along K, stride offset K / 8 * 128
// between 8-row groups); the instruction descriptor marks the operand MN-major.
__host__ __device__ constexpr uint32_t mnmaj_off(int r, int k, int K) {
  return (uint32_t)((((r >> 3) * (K >> 3)) + (k >> 3)) * 128 + (k & 7) * 16 + (r & 7) * 2);
}

// Shared-memory matrix descriptor: start address, leading / stride byte
// offsets (all in 16-byte units), descriptor version 1 (bits 46-47), no swizzle.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}
// Descriptor of a K-major no-swizzle operand with K columns, starting at K step kk (16 columns each).
__device__ __forceinline__ uint64_t kmaj_desc(uint32_t base, int K, int kk) {
  return sdesc(base + (uint32_t)kk * 256u, 128u, (uint32_t)(K >> 3) * 128u);
}

// Instruction descriptor of kind::f16: bf16 A and B, fp32 D, M x N; A and B
// K-major unless a_mn / b_mn mark them MN-major (bits 15 and 16).
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn = false,
                                                      bool b_mn = false) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Allocate ncols TMEM columns (a power of two >= 32); one whole warp executes
// it.  The base address is written to *slot (shared memory).
__device__ __forceinline__ void tmem_alloc(uint32_t slot_saddr, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_saddr),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// D (TMEM) = A * B^T (+ D when accumulate): one MMA, issued by one thread.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on the mbarrier when every MMA this thread issued so far has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar_saddr) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar_saddr)
               : "memory");
}

__device__ __forceinline__ void fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Generic-proxy shared-memory writes made visible to the tensor cores (async proxy).
__device__ __forceinline__ void fence_smem_to_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 32 consecutive 32-bit columns of this thread's lane (warp-wide, .sync.aligned).
// The registers are not valid until tmem_wait_ld(r) has run on them.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
// Wait for this thread's outstanding TMEM loads.  The registers of `r` are
// in/out operands, so no use of them can be scheduled before the wait.
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]),
                 "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                 "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]),
                 "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}

// 16 consecutive 32-bit columns of this thread's lane; valid after tmem_wait_ld16(r).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld16(uint32_t (&r)[16]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
}

}  // namespace tc
}  // namespace dl
