// wmtp_tc.cuh -- 5th-generation tensor-core (tcgen05) wrappers for sm_103a:
// tensor-memory allocation, MMA issue from shared-memory descriptors,
// completion through mbarriers, and tensor-memory loads/stores.
//
// Shared-memory operands use the no-swizzle canonical layout built from 8x8
// "core matrices" (8 rows of 16 bytes, 128 contiguous bytes):
//   K-major operand (rows x K): byte offset of (row, k) =
//       (row / 8) * SBO + (k / 8) * LBO + (row % 8) * 16 + (k % 8) * 2
//   MN-major operand (K x N, N contiguous): byte offset of (n, k) =
//       (n / 8) * SBO + (k / 8) * LBO + (k % 8) * 16 + (n % 8) * 2
// i.e. LBO steps between core matrices along K, SBO along M/N.  These
// encodings were checked on the device against exact integer products
// before use.
#pragma once

#include <stdint.h>

namespace wmtp {

// Shared-memory matrix descriptor: start address, LBO, SBO (all >> 4),
// descriptor version 1 (bit 46), no swizzle, base offset 0.
__device__ __forceinline__ uint64_t tc_smem_desc(uint32_t smem_addr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = (uint64_t)((smem_addr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    return d;
}

// Descriptor of an operand in the 128-byte-swizzled canonical layout
// (swizzle mode 2 in bits 61-63): 8-row atoms of 128-byte rows, 1024-byte
// aligned, whose 16-byte chunks are XORed with the row within the atom (the
// layout a 128-byte-swizzle TMA box writes).  K-major: SBO = stride between
// 8-row atoms, steps along K inside an atom advance the start address by
// 32 bytes per 16 elements; MN-major: LBO = stride between 64-element blocks
// along M/N, SBO = stride between 8-row atoms along K.  Checked on the device
// against exact integer products before use.
__device__ __forceinline__ uint64_t tc_smem_desc_sw128(uint32_t smem_addr, uint32_t lbo, uint32_t sbo) {
    return tc_smem_desc(smem_addr, lbo, sbo) | ((uint64_t)2 << 61);
}

// Instruction descriptor for kind::f16 with bf16 A and B, fp32 D.
// b_mn_major: B stored N-contiguous (transposed).
__host__ __device__ constexpr uint32_t tc_idesc_bf16(int M, int N, int b_mn_major) {
    return (1u << 4)                      // D: f32
           | (1u << 7)                    // A: bf16
           | (1u << 10)                   // B: bf16
           | ((uint32_t)b_mn_major << 16)  // B major-ness
           | ((uint32_t)(N >> 3) << 17)   // N / 8
           | ((uint32_t)(M >> 4) << 24);  // M / 16
}

// Allocates `ncols` tensor-memory columns (whole warp); the base address is
// written to shared memory at `dst`.
__device__ __forceinline__ void tc_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tc_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]; issued by one thread.
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]: A (M rows = lanes) from tensor memory,
// two 16-bit elements per 32-bit column, K = 16 per instruction (8 columns);
// checked on the device against exact integer products before use.
__device__ __forceinline__ void tc_mma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                               uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrives once on `mbar` when every tcgen05 operation issued so far by this
// thread has completed.
__device__ __forceinline__ void tc_commit(uint32_t mbar_smem) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(mbar_smem)
        : "memory");
}

// 32 consecutive 32-bit columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tc_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tc_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

}  // namespace wmtp
