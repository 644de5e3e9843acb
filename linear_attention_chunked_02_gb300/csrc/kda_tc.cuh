// kda_tc.cuh -- sm_103a tensor-core (tcgen05) and tensor-memory helpers.
//
// Thin inline-PTX wrappers for the fifth-generation tensor-core path:
//   * tensor memory (TMEM) allocation, owned by one warp of the CTA;
//   * tcgen05.mma of kind::tf32 with both operands in shared memory, described
//     by 64-bit matrix descriptors, and the FP32 accumulator in TMEM;
//   * tcgen05.commit onto an mbarrier (completion of the MMAs issued so far);
//   * tcgen05.ld of accumulator rows into registers.
// Operand tiles are K-major with the 128-byte swizzle: row r of a tile is 128
// bytes (32 TF32 values) at byte r * 128 of a 1024-byte aligned buffer, its
// 16-byte chunk c stored at chunk position c ^ (r & 7); eight rows form one
// 1024-byte swizzle atom, and atoms follow each other along M (or N).
#pragma once

#include <stdint.h>

namespace kda {
namespace tc {

// ------------------------------------------------------------ descriptors
// Shared-memory matrix descriptor of a K-major, 128-byte-swizzled tile whose
// first row starts at shared address `addr` (1024-byte aligned for the first
// K step; later K steps of 8 TF32 values advance the start by 32 bytes inside
// the atom).  Fields: start address >> 4 (bits 0-13), leading byte offset >> 4
// (bits 16-29; unused by this layout, set to 1), stride byte offset >> 4
// (bits 32-45: 1024 bytes between 8-row groups), descriptor version 1 (bits
// 46-47), base offset 0 (bits 49-51), layout type 2 = 128-byte swizzle (bits
// 61-63).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr) {
    uint64_t d = 0;
    d |= uint64_t((addr & 0x3FFFFu) >> 4);
    d |= uint64_t(16u >> 4) << 16;
    d |= uint64_t(1024u >> 4) << 32;
    d |= uint64_t(1) << 46;
    d |= uint64_t(2) << 61;
    return d;
}

// Instruction descriptor of tcgen05.mma kind::tf32: FP32 accumulator (bits
// 4-5 = 1), A and B TF32 (bits 7-9 and 10-12 = 2), both K-major (bits 15, 16 =
// 0), N >> 3 in bits 17-22, M >> 4 in bits 24-28; dense, no negation.
template <int M, int N>
__host__ __device__ constexpr uint32_t idesc_tf32() {
    static_assert(M == 64 || M == 128, "M of one CTA");
    static_assert(N % 16 == 0 && N >= 16 && N <= 256, "N");
    return (1u << 4) | (2u << 7) | (2u << 10) | (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

// ------------------------------------------------------------------ TMEM
// Allocate `ncols` TMEM columns (power of two >= 32) for this CTA; the whole
// warp executes it, the address lands in shared memory at `slot`.
__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// ------------------------------------------------------------------- MMA
// D[tmem] (+)= A[smem] * B[smem]^T, one K step (8 TF32 values).
__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(uint32_t(accumulate))
        : "memory");
}
// Arrive once on the mbarrier when every tcgen05 operation this thread issued
// so far has completed.
__device__ __forceinline__ void commit(uint32_t mbar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar)
                 : "memory");
}
__device__ __forceinline__ void fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ------------------------------------------------------------- TMEM loads
// 16 consecutive 32-bit columns of the warp's TMEM lane (lane = warp quarter
// base + lane id; `taddr` carries the quarter base in bits 16-31).
__device__ __forceinline__ void ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

}  // namespace tc
}  // namespace kda
