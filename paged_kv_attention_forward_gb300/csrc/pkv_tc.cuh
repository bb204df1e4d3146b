// pkv_tc.cuh -- inline-PTX wrappers for the 5th-generation tensor cores (sm_100 family):
// tensor-memory allocation, tcgen05.mma (kind::f16, one CTA), its commit to an mbarrier,
// tcgen05.ld of accumulator columns, the tcgen05 fences, and the shared-memory matrix
// and instruction descriptors the MMA reads its operands through.
//
// Operand layouts used here (16-bit elements, 128-byte swizzle, the layout a TMA tile
// load with CU_TENSOR_MAP_SWIZZLE_128B writes):
//  * K-major: row r of the operand (an M or N index) holds 64 consecutive K elements in
//    128 bytes; 8 rows form a 1024-byte swizzle atom; atoms of 8 rows follow each other
//    at `sbo` bytes.  A K-step of 16 elements starts 32 bytes further in (within one atom
//    row), so one 64-element half of K is addressed by a start address alone.
//  * MN-major: row k of the stored tile (a K index) holds 64 consecutive M (or N)
//    elements in 128 bytes; 8 K rows form an atom; `sbo` is the byte distance between
//    groups of 8 K rows and `lbo` the distance between 64-element M blocks.
#pragma once

#include <cstdint>

namespace pkv {
namespace tc {

// ---- tensor memory ----------------------------------------------------------
// Allocate `ncols` columns (a power of two >= 32) of this CTA's tensor memory; the base
// address is written to *dst (shared memory).  Executed by one whole warp.
__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "r"(ncols)
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

// ---- fences -----------------------------------------------------------------
__device__ __forceinline__ void fence_before_sync()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void fence_after_sync()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// generic-proxy shared-memory writes -> visible to the async proxy (the MMA's operand reads)
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- descriptors ------------------------------------------------------------
// Shared-memory matrix descriptor, 128-byte swizzle: start address, leading and stride
// byte offsets (all >> 4), the fixed version field 0b001 at bit 46, swizzle mode 2 at
// bits 61-63.  The start of a swizzle atom must be 1024-byte aligned; a start address
// inside an atom row (a K-step) keeps base offset 0.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1u << 46;
    d |= (uint64_t)2u << 61;
    return d;
}

// Instruction descriptor of tcgen05.mma kind::f16: bf16 A and B, fp32 accumulator,
// M x N, A / B K-major (0) or MN-major (1).
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, int a_mn_major, int b_mn_major)
{
    return (1u << 4)                              // D: f32
           | (1u << 7)                            // A: bf16
           | (1u << 10)                           // B: bf16
           | ((uint32_t)a_mn_major << 15)         // A major-ness
           | ((uint32_t)b_mn_major << 16)         // B major-ness
           | ((uint32_t)(N >> 3) << 17)           // N / 8
           | ((uint32_t)(M >> 4) << 24);          // M / 16
}

// ---- MMA --------------------------------------------------------------------
// D[tmem] (+)= A(smem desc) x B(smem desc); issued by one thread.
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

// Arrive (once) on `bar` when every MMA this thread issued before has completed.
__device__ __forceinline__ void mma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(bar)))
                 : "memory");
}

// ---- accumulator loads --------------------------------------------------------
// Thread t of warp w (w % 4 selects the 32-lane quarter) reads lane 32 (w % 4) + t,
// columns col .. col + 15 of the address's lane base.  The registers are valid only
// after tmem_wait(): read them through it.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

// Wait for this thread's tcgen05.ld results, then pass the loaded registers through an
// empty asm after the wait, so no use of them can be scheduled before it.
template <int N>
__device__ __forceinline__ void tmem_wait(uint32_t (&r)[N])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < N; ++i)
        asm volatile("" : "+r"(r[i]));
}

// The same for several loads in flight at once (one wait for all of them).
template <int T, int N>
__device__ __forceinline__ void tmem_wait(uint32_t (&r)[T][N])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int t = 0; t < T; ++t)
#pragma unroll
        for (int i = 0; i < N; ++i)
            asm volatile("" : "+r"(r[t][i]));
}

}  // namespace tc
}  // namespace pkv
