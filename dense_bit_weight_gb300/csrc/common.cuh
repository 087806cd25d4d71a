// common.cuh -- small device helpers shared by the kernel translation units.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/dbw_gemm.h"

namespace dbw {

// bf16 pair (packed in one 32-bit word, element 0 in the low half) -> two fp32.
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// fp32 -> bf16, round to nearest even (hardware cvt.rn).
__device__ __forceinline__ uint16_t f32_to_bf16_rn(float x)
{
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// Two fp32 -> packed bf16x2 (lo in the low half), round to nearest even.
__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// 128-bit streaming load that bypasses L1 allocation (weights are read once).
__device__ __forceinline__ uint4 ld_stream_v4(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// 128-bit read-only load through L1 (activations are reused by every row).
__device__ __forceinline__ uint4 ld_ro_v4(const void *p)
{
    return __ldg(reinterpret_cast<const uint4 *>(p));
}

// The gated-MLP epilogue: silu(g) * u with silu(x) = x / (1 + e^-x), in fp32
// (IEEE division, so a huge negative g gives -0, not NaN).
__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.f + __expf(-g)) * u; }

// The bias epilogues: x + b, then the epilogue's activation (relu, silu, or
// the exact erf form of gelu), in fp32.
__device__ __forceinline__ float bias_act(float x, float b, int epi)
{
    x += b;
    if (epi == GEMM_EPI_BIAS_RELU) return fmaxf(x, 0.f);
    if (epi == GEMM_EPI_BIAS_SILU) return x / (1.f + __expf(-x));
    if (epi == GEMM_EPI_BIAS_GELU) return 0.5f * x * (1.f + erff(x * 0.70710678118654752f));
    return x;
}

// Whether an epilogue adds a bias (plain or with an activation).
__host__ __device__ constexpr bool epi_has_bias(int epi)
{
    return epi == GEMM_EPI_BIAS || (epi >= GEMM_EPI_BIAS_RELU && epi <= GEMM_EPI_BIAS_GELU);
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

}  // namespace dbw
