// pi_umma.cuh -- 5th-generation tensor-core (tcgen05) building blocks for sm_103a.
//
// Operand tiles live in shared memory in the canonical 128-byte-swizzled layouts:
//   K-major  (rows of the contraction dimension K contiguous): an 8-row x 128-byte atom
//            holds 8 rows x 64 16-bit elements; the 16-byte chunk c of row r sits at
//            chunk position c ^ (r % 8). Atoms of consecutive 8-row groups are SBO apart.
//   MN-major (rows of the M or N dimension contiguous): the same atom holds 8 K-indices x
//            64 MN-elements; atoms are LBO apart along MN and SBO apart along K.
// Atoms start on 1024-byte boundaries, so the swizzle is a function of the address.
// Accumulators are fp32 in tensor memory (TMEM): lane = output row, column = output column.
#pragma once

#include <cuda_bf16.h>

#include "pi_async.cuh"

namespace pi {

// ---------------------------------------------------------------- descriptors ----------------

// Shared-memory matrix descriptor: start address, leading / stride byte offsets, the
// fixed 0b001 at bits 46-48, and the 128-byte swizzle mode (2) at bits 61-63.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo)
{
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor of kind::f16 with an fp32 accumulator. ab_bf16: both operands
// bf16 (else both fp16). a_mn / b_mn: operand stored MN-major (else K-major).
__host__ __device__ constexpr uint32_t f16_idesc(int ab_bf16, int a_mn, int b_mn, int M, int N)
{
    return (1u << 4) | ((uint32_t)ab_bf16 << 7) | ((uint32_t)ab_bf16 << 10) | ((uint32_t)a_mn << 15) |
           ((uint32_t)b_mn << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Byte offset of 16-byte chunk c (0..7) of row r inside a run of 128-byte-swizzled atoms
// whose 8-row groups are consecutive (1024 bytes apart).
__device__ __forceinline__ uint32_t sw128_off(uint32_t r, uint32_t c)
{
    return (r >> 3) * 1024u + (r & 7u) * 128u + ((c ^ (r & 7u)) << 4);
}

// ---------------------------------------------------------------- TMEM -----------------------

// One full warp: allocate `ncols` (power of two, 32..512) TMEM columns; the address is
// written to *dst (shared memory).
__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// ---------------------------------------------------------------- MMA ------------------------

// D[tmem] (+)= A * B, one elected thread. accum = false overwrites D.
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         bool accum)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"((uint32_t)accum)
        : "memory");
}

// Arrive once on `bar` when every tcgen05 operation this thread issued so far is done.
__device__ __forceinline__ void umma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// 16 consecutive fp32 columns of this thread's TMEM lane (warp w reads lanes 32*(w%4)..+31).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// ---------------------------------------------------------------- cp.async -------------------

// 16-byte global -> shared copy (L2 only); src_bytes = 0 fills the 16 bytes with zeros.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Arrive on `bar` once every cp.async this thread issued so far has completed (the barrier's
// expected count includes this arrival).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t *bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Named barrier over `n` threads (id 1..15).
__device__ __forceinline__ void named_sync(int id, int n)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// ---------------------------------------------------------------- activation split ----------

// x = hi + lo with hi, lo in the weights' 16-bit type: the pair carries ~16 more bits of x
// than hi alone, so a tensor-core product with exact 16-bit weights keeps fp32-level accuracy.
template <int WT>
__device__ __forceinline__ void split16(float x, uint16_t &hi, uint16_t &lo);

// fp32 operands never take the 16-bit tensor-core paths; this only completes the set
template <>
__device__ __forceinline__ void split16<DT_F32>(float, uint16_t &hi, uint16_t &lo)
{
    hi = 0;
    lo = 0;
}

template <>
__device__ __forceinline__ void split16<DT_BF16>(float x, uint16_t &hi, uint16_t &lo)
{
    const __nv_bfloat16 h = __float2bfloat16_rn(x);
    const __nv_bfloat16 l = __float2bfloat16_rn(x - __bfloat162float(h));
    hi = __bfloat16_as_ushort(h);
    lo = __bfloat16_as_ushort(l);
}

template <>
__device__ __forceinline__ void split16<DT_F16>(float x, uint16_t &hi, uint16_t &lo)
{
    const __half h = __float2half_rn(x);
    const __half l = __float2half_rn(x - __half2float(h));
    hi = __half_as_ushort(h);
    lo = __half_as_ushort(l);
}

}  // namespace pi
