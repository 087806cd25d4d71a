// frag.cuh -- device helpers shared by the kernels built on warp-level MMAs
// (mma.sync fragments) and 1-D bulk copies.
#pragma once

#include <stdint.h>

namespace dbw {

// bf16x2 (128 + q_p, 128 + q_{p+4}) from nibble pair p of a packed 4-bit
// word: 128 + q is exact in bf16 as the bit pattern 0x4300 | q.
__device__ __forceinline__ uint32_t pair128(uint32_t x, int p)
{
    return ((x >> (4 * p)) & 0x000F000Fu) | 0x43004300u;
}

// d += A B on the warp-level tensor path: mma.sync.m16n8k16, bf16 operands
// (A: 16 x 16 in four registers per lane, B: 16 x 8 in two), fp32 accumulator.
__device__ __forceinline__ void mma_acc(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Ask L2 for `bytes` (a multiple of 16) at `src` without writing shared memory.
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(src)), "r"(bytes)
                 : "memory");
}

// Global -> shared 1-D bulk copy (16-byte aligned ends, size a multiple of
// 16), its bytes counted on the mbarrier `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
                 : "memory");
}

}  // namespace dbw
