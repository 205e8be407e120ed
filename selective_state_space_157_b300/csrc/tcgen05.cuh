// tcgen05.cuh -- the fifth-generation tensor core instructions of sm_100-family
// GPUs (here sm_103a), as inline PTX: tensor-memory (TMEM) allocation,
// tcgen05.mma with fp16 operands staged in shared memory and an fp32
// accumulator in TMEM, completion through an mbarrier, and TMEM loads.
//
// Operand layout in shared memory: K-major without swizzle, as 8 x 16-byte
// "core matrices" (8 rows of 8 fp16 along K). Core matrix (i, j) holds rows
// 8i..8i+7 and k 8j..8j+7 and sits at ((i * K/8) + j) * 128 bytes, so the
// K-direction neighbour is 128 bytes on (the descriptor's leading byte
// offset) and the next 8 rows K/8 * 128 bytes on (its stride byte offset).
// Checked on a B300 against a CPU product (M = 64 and 128, K = 16 and 64).
//
// Accumulator layout in TMEM (one column per output column): for M = 128,
// row r is lane r; for M = 64, rows 16w .. 16w+15 are lanes 32w .. 32w+15.
// Warp w of a CTA may read lanes 32(w % 4) .. 32(w % 4) + 31 only.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "tma.cuh"

namespace selscan {

// Index (in fp16 elements) of element (r, k) of a K-major tile with K
// columns, in core-matrix order.
__host__ __device__ __forceinline__ int core_index(int r, int k, int K)
{
    return (((r >> 3) * (K >> 3) + (k >> 3)) << 6) + ((r & 7) << 3) + (k & 7);
}

// Shared-memory matrix descriptor: start address, leading and stride byte
// offsets (in 16-byte units), descriptor version 1, no swizzle.
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFF);
    d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
    d |= (uint64_t)1 << 46;
    return d;
}

// Descriptor of a K-major tile with K columns, advanced to k-step kk (16
// columns per MMA instruction).
__device__ __forceinline__ uint64_t umma_tile_desc(const void *tile, int K, int kk)
{
    return umma_desc(smem_u32(tile) + (uint32_t)kk * 256u, 128u, (uint32_t)(K >> 3) * 128u);
}

// Instruction descriptor of tcgen05.mma kind::f16: fp16 A and B, fp32
// accumulator, both operands K-major, shape M x N (x 16).
__host__ __device__ constexpr uint32_t umma_idesc_f16(int M, int N)
{
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Allocates ncols TMEM columns (a power of two >= 32); one full warp calls
// it. The TMEM address is written to *dst (shared memory).
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

__device__ __forceinline__ void tc_fence_after()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_before()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

// D (TMEM) = A * B^T (+ D when accumulate): one instruction, K = 16.
__device__ __forceinline__ void umma_f16(uint32_t dtmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         bool accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(dtmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"((int)accumulate)
        : "memory");
}

// Arrives on *bar once every MMA this thread issued before has completed.
__device__ __forceinline__ void umma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// Starts loading 16 consecutive fp32 columns of this thread's TMEM lane
// (warp-wide); the values are usable after tmem_wait_ld().
__device__ __forceinline__ void tmem_ld16_async(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
                   "=r"(r[15])
                 : "r"(taddr)
                 : "memory");
}

// Waits for every TMEM load this thread started.
__device__ __forceinline__ void tmem_wait_ld()
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Loads 16 consecutive fp32 columns of this thread's TMEM lane (warp-wide),
// and waits for them.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
                   "=r"(r[15])
                 : "r"(taddr)
                 : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i)
        v[i] = __uint_as_float(r[i]);
}

} // namespace selscan
