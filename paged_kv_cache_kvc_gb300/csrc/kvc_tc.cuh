// Fifth-generation tensor cores (tcgen05) on sm_103a: tensor-memory (TMEM)
// allocation, the single-thread MMA with operands in shared memory and the
// accumulator in TMEM, its completion barrier, and TMEM loads / stores.
//
// Operand descriptors (64 bits, one per MMA operand in shared memory):
//   bits  0..13  start address >> 4
//   bits 16..29  leading-dimension byte offset >> 4
//   bits 32..45  stride-dimension byte offset >> 4
//   bits 46..47  descriptor version, 1 for tcgen05
//   bits 49..51  base offset (0: every swizzle atom 1024-byte aligned)
//   bit  52      leading-dimension offset mode (0: relative)
//   bits 61..63  swizzle: 0 none, 2 128-byte, 4 64-byte, 6 32-byte
// With the 128-byte swizzle an atom is 8 rows of 128 bytes (1024 bytes); in
// row r, 16-byte chunk c is stored at chunk c ^ (r mod 8).  Two operand forms:
//   K-major  (the reduction index contiguous in a row): rows are M (or N)
//            indices, an 8-row group every SBO bytes; LBO is unused.  A step
//            of 16 bf16 along K inside an atom adds 32 bytes to the start.
//   MN-major (the M or N index contiguous in a row): rows are K indices, an
//            8-row group every SBO bytes; the next 64 M (or N) indices (the
//            next 128-byte column band) are LBO bytes further.
//
// Instruction descriptor of kind::f16 (32 bits):
//   bits  4..5   accumulator type: 1 = f32
//   bits  7..9   A type: 0 f16, 1 bf16;  bits 10..12 B type (same)
//   bit  15      A is MN-major;  bit 16  B is MN-major
//   bits 17..22  N >> 3;  bits 24..28  M >> 4
//
// Accumulator of an M = 128 MMA: row i in TMEM lane i, column j in column
// base + j (fp32).  A warp reaches only its quarter of the lanes:
// 32 * (warp mod 4) .. + 31.  TMEM addresses: lane << 16 | column.
#pragma once
#include <cstdint>

namespace kvc {

enum : uint32_t { kSwizzleNone = 0, kSwizzle128B = 2, kSwizzle64B = 4, kSwizzle32B = 6 };

__host__ __device__ constexpr uint64_t tc_smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t swizzle)
{
    return static_cast<uint64_t>((addr >> 4) & 0x3FFFu) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
           (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (uint64_t(1) << 46) |
           (static_cast<uint64_t>(swizzle & 7u) << 61);
}

__host__ __device__ constexpr uint32_t tc_idesc_f16(int M, int N, bool bf16, bool a_mn_major, bool b_mn_major)
{
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) | ((a_mn_major ? 1u : 0u) << 15) |
           ((b_mn_major ? 1u : 0u) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
           (static_cast<uint32_t>(M >> 4) << 24);
}

// The same descriptor with its start address moved by `bytes` (a multiple of 16; the
// 14-bit field holds every shared-memory address, so the add never carries out of it).
__host__ __device__ constexpr uint64_t tc_desc_advance(uint64_t desc, uint32_t bytes)
{
    return desc + (bytes >> 4);
}

// Byte offset of 16-byte chunk `ch` of 128-byte row `row` inside a run of
// 128-byte-swizzled atoms (the layout TMA writes with the 128-byte swizzle).
__host__ __device__ constexpr uint32_t sw128(uint32_t row, uint32_t ch)
{
    return row * 128u + (((ch ^ row) & 7u) << 4);
}

// ------------------------------------------------------------------ TMEM allocation (whole warp)
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// ------------------------------------------------------------------ ordering around thread synchronisation
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// ------------------------------------------------------------------ MMA (one thread issues)
// D[tmem] (+)= A[smem desc] * B[smem desc]; accumulate = 0 overwrites D.
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on the mbarrier when every MMA this thread issued so far has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// The same two, called by every lane of a converged warp with the same operands: one
// elected lane issues.  Computing the descriptors warp-wide keeps them warp-uniform,
// and the elected lane is the same for an MMA and the commit that tracks it.
__device__ __forceinline__ void tc_mma_f16_warp(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// The MMA with its A operand in tensor memory (warp-wide, one elected lane issues): row i of
// A in lane i, 16-bit elements k = 2c, 2c + 1 in the low and high halves of column a_tmem + c
// (K-major); B from shared memory as above.
__device__ __forceinline__ void tc_mma_f16_tmem_a_warp(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                       uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
        ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tc_commit_warp(uint32_t bar)
{
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}"
        ::"r"(bar)
        : "memory");
}

// ------------------------------------------------------------------ TMEM <-> registers (whole warp)
// Thread i of the warp reads lane (taddr's lane + i), 32 consecutive columns.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

// Wait for this thread's TMEM loads.  The registers are named as operands so
// that no use of them is scheduled before the wait.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[32])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                   "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                   "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};"
        ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
          "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
          "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]),
          "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ------------------------------------------------------------------ softmax arithmetic
__device__ __forceinline__ float max3f(float a, float b, float c)
{
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

}  // namespace kvc
