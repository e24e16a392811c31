// tc.cuh -- inline-PTX access to the 5th-generation tensor cores (tcgen05)
// and tensor memory (TMEM) of sm_103a, as the forward's Gram kernel uses them:
// one CTA, one elected thread issuing bf16 MMAs whose operands sit in shared
// memory in the K-major 128-byte-swizzle layout, fp32 accumulators in TMEM,
// read back by each warp from its own quarter of the TMEM lanes.
#pragma once

#include "common.cuh"

namespace dlrm {
namespace tc {

// ---- tensor memory ----------------------------------------------------------
// Allocate `ncols` columns (a power of two >= 32) of TMEM for this CTA; a whole
// warp executes it and the base address lands in shared memory at *dst.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst)),
                 "r"(ncols)
                 : "memory");
}

// This CTA will not allocate again (lets other CTAs on the SM allocate).
__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Order tcgen05 operations around a thread barrier.
__device__ __forceinline__ void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Make this thread's ordinary shared-memory stores visible to the tensor
// core, which reads its operands through the async proxy.
__device__ __forceinline__ void fence_smem_for_mma() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// ---- descriptors ------------------------------------------------------------
// Shared-memory matrix descriptor of a K-major bf16 operand in the 128-byte
// swizzle layout: each row holds 64 elements (128 B) of K; the 16-byte chunk c
// of row r sits at chunk position c ^ (r % 8); rows are 128 B apart, 8-row
// groups 1024 B apart (stride byte offset); the layout's base is 1024-byte
// aligned.  Moving `saddr` by 32 B selects the next 16 elements of K.
__device__ __forceinline__ uint64_t desc_kmajor_sw128(uint32_t saddr)
{
    return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4)  // start address
           | (static_cast<uint64_t>(1) << 16)               // leading byte offset (not used with this swizzle)
           | (static_cast<uint64_t>(1024 >> 4) << 32)       // stride byte offset: next 8 rows
           | (static_cast<uint64_t>(1) << 46)               // descriptor version of tcgen05
           | (static_cast<uint64_t>(2) << 61);              // 128-byte swizzle
}

// Instruction descriptor of kind::f16: bf16 A and B, both K-major, fp32
// accumulator, M x N tile, dense, no negation.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N)
{
    return (1u << 4)                                   // D: fp32
           | (1u << 7)                                 // A: bf16
           | (1u << 10)                                // B: bf16
           | (static_cast<uint32_t>(N >> 3) << 17)     // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24);    // M / 16
}

// ---- MMA ----------------------------------------------------------------------
// D[tmem] (+)= A * B^T, A: M x 16 and B: N x 16 bf16 from shared memory.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when every MMA this thread issued before has completed
// (results in TMEM, shared-memory operands no longer read).
__device__ __forceinline__ void commit(uint64_t* bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_addr(bar))
                 : "memory");
}

// ---- TMEM -> registers --------------------------------------------------------
// Thread i of the warp receives 32 consecutive 32-bit columns of TMEM lane
// (lane field of taddr) + i.  A warp may read only the 32 lanes of its own
// quarter: lanes 32*(warp % 4) .. +31.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

}  // namespace tc
}  // namespace dlrm
