// 5th-generation tensor core (tcgen05) building blocks, in inline PTX: tensor-memory allocation,
// shared-memory matrix descriptors for K-major tiles with the 128-byte swizzle, the dense bf16 MMA
// with an fp32 accumulator in tensor memory, its commit to an mbarrier, and the tensor-memory loads
// of the epilogue.
#pragma once
#include <cstdint>

namespace verkv {

__device__ __forceinline__ unsigned umma_smem_u32(const void* p) { return (unsigned)__cvta_generic_to_shared(p); }

// Byte offset of element (row, k) of a K-major bf16 tile of `rows` rows and 128 K elements stored for
// the 128-byte swizzle: two K halves of 64 elements, each [rows / 8][8 rows][128 B], the 16-byte
// chunk index XORed with row % 8.  The tile must start on a 1024-byte boundary.
__device__ __forceinline__ unsigned umma_sw128_offset(int row, int k, int rows)
{
    const int half = k >> 6, kk = k & 63;
    return (unsigned)(half * (rows / 8) * 1024 + (row >> 3) * 1024 + (row & 7) * 128 +
                      (((kk >> 3) ^ (row & 7)) << 4) + (kk & 7) * 2);
}

// Shared-memory matrix descriptor: start address, stride of 1024 B between 8-row groups, 128-byte
// swizzle (the leading byte offset is unused for swizzled K-major tiles).
__device__ __forceinline__ uint64_t umma_desc_sw128(unsigned smem_addr)
{
    uint64_t d = (uint64_t)((smem_addr >> 4) & 0x3FFFu);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor of kind::f16: bf16 A and B (K-major), fp32 D, M x N.
__host__ __device__ constexpr unsigned umma_idesc_bf16_f32(int M, int N)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((unsigned)(N >> 3) << 17) | ((unsigned)(M >> 4) << 24);
}

// Instruction descriptor of kind::f16: fp16 A and B (K-major), fp32 D, M x N.
__host__ __device__ constexpr unsigned umma_idesc_f16_f32(int M, int N)
{
    return (1u << 4) | ((unsigned)(N >> 3) << 17) | ((unsigned)(M >> 4) << 24);
}

// Start of K step ks (16 elements) of a tile laid out by umma_sw128_offset.
__device__ __forceinline__ unsigned umma_kstep_offset(int ks, int rows)
{
    return (unsigned)((ks >> 2) * (rows / 8) * 1024 + (ks & 3) * 32);
}

__device__ __forceinline__ void umma_alloc(unsigned* dst_smem, unsigned ncols)   // one full warp
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(umma_smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void umma_dealloc(unsigned taddr, unsigned ncols)   // the allocating warp
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// D[tmem] (+)= A * B^T (kind::f16: the operand types are those of the instruction descriptor), one
// elected thread.
__device__ __forceinline__ void umma_mma(unsigned tmem_d, uint64_t adesc, uint64_t bdesc, unsigned idesc, bool acc)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
                 "l"(adesc), "l"(bdesc), "r"(idesc), "r"((unsigned)acc)
                 : "memory");
}

// Arrive on the mbarrier once all MMAs issued so far by this thread have completed.
__device__ __forceinline__ void umma_commit(unsigned long long* bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     umma_smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void umma_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void umma_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 16 consecutive fp32 columns of this thread's tensor-memory lane (warp w of the block reads lanes
// 32 (w % 4) .. 32 (w % 4) + 31).
__device__ __forceinline__ void umma_ld16(unsigned taddr, float (&v)[16])
{
    unsigned r[16];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
}

}  // namespace verkv
