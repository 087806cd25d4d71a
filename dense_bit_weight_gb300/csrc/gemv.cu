// gemv.cu -- CUDA-core weight-streaming kernels for small M (decode).
//
// One warp owns one weight row n at a time and walks K in 16-byte chunks
// (lane l takes chunks l, l+32, ...), so each warp instruction reads 512
// contiguous bytes of the row; the weights are read with no-L1-allocate
// loads, the activations through L1 (every row reuses them).  The K sum is
// finished with a butterfly of warp shuffles and lane 0 writes the output.
// This is the decode GEMV of the hk-dsl PyPI page ("Results", kernels inside
// the engines: "decode GEMV, 1-32 tokens"), with the cross-lane reduction of
// the FlyDSL prebuilt kernels guide §2 (XOR-shuffle warp reduction).
//
// For M larger than the per-pass row count the kernel makes one pass over the
// weight row per group of rows (the tcgen05 kernels serve those shapes).
// Fused epilogues: EPI = 1 adds bias[n] to the fp32 sum and applies the
// epilogue's activation (none, relu, silu or gelu); EPI = 2 has the warp take
// the weight rows n (gate) and N + n (up) together and store silu(gate) * up.
#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace dbw {
namespace {

constexpr int kWarps = 8;

template <int MT, int U, int EPI>
__global__ void __launch_bounds__(kWarps * 32)
k_gemv_bf16(const uint16_t *__restrict__ A, const uint16_t *__restrict__ B,
            uint16_t *__restrict__ C, int M, int N, int K, int64_t lda, int64_t ldb, int64_t ldc,
            const uint16_t *__restrict__ bias, int epi)
{
    ptx::pdl_wait();
    ptx::pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int chunks = K >> 3;  // 8 bf16 per 16-byte chunk
    constexpr int NR = EPI == 2 ? 2 : 1;   // weight rows per output column
    for (int n = blockIdx.x * kWarps + (threadIdx.x >> 5); n < N; n += gridDim.x * kWarps) {
        const uint16_t *brow[NR];
#pragma unroll
        for (int r = 0; r < NR; ++r) brow[r] = B + (int64_t)(n + r * N) * ldb;
        for (int m0 = 0; m0 < M; m0 += MT) {
            float acc[NR][MT];
#pragma unroll
            for (int r = 0; r < NR; ++r)
#pragma unroll
                for (int i = 0; i < MT; ++i) acc[r][i] = 0.f;
            for (int c0 = lane; c0 < chunks; c0 += 32 * U) {
                uint4 bv[NR][U];
#pragma unroll
                for (int r = 0; r < NR; ++r)
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        const int c = c0 + 32 * u;
                        bv[r][u] = c < chunks ? ld_stream_v4(brow[r] + (int64_t)c * 8) : make_uint4(0, 0, 0, 0);
                    }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int c = c0 + 32 * u;
                    if (c >= chunks) break;
#pragma unroll
                    for (int i = 0; i < MT; ++i) {
                        if (m0 + i >= M) break;
                        const uint4 av = ld_ro_v4(A + (int64_t)(m0 + i) * lda + (int64_t)c * 8);
                        const uint32_t aw[4] = {av.x, av.y, av.z, av.w};
#pragma unroll
                        for (int r = 0; r < NR; ++r) {
                            const uint32_t bw[4] = {bv[r][u].x, bv[r][u].y, bv[r][u].z, bv[r][u].w};
                            float s = acc[r][i];
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                s = fmaf(bf16lo(aw[j]), bf16lo(bw[j]), s);
                                s = fmaf(bf16hi(aw[j]), bf16hi(bw[j]), s);
                            }
                            acc[r][i] = s;
                        }
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < MT; ++i) {
                float v = warp_sum(acc[0][i]);
                if (EPI == 1) v = bias_act(v, bf16lo(bias[n]), epi);
                if (EPI == 2) v = silu_mul(v, warp_sum(acc[NR - 1][i]));
                if (lane == 0 && m0 + i < M) C[(int64_t)(m0 + i) * ldc + n] = f32_to_bf16_rn(v);
            }
        }
    }
}

// W4A16: each lane takes 16 bytes of packed weights = 32 consecutive k, which
// never straddle a quantisation group (group is a multiple of 32).  With
// w = (q - z) * s for the whole chunk,
//     sum_k a_k w_k = s * (sum_k a_k q_k - z * sum_k a_k),
// exact in real arithmetic; here each partial sum is fp32.
template <int MT>
__global__ void __launch_bounds__(kWarps * 32)
k_gemv_w4a16(const uint16_t *__restrict__ A, const uint32_t *__restrict__ Bq,
             const uint16_t *__restrict__ S, const uint8_t *__restrict__ Z,
             uint16_t *__restrict__ C, int M, int N, int K, int group)
{
    ptx::pdl_wait();
    ptx::pdl_launch_dependents();
    constexpr int U = 4;
    const int lane = threadIdx.x & 31;
    const int chunks = K >> 5;      // 32 k (16 bytes of Bq) per chunk
    const int groups = K / group;
    for (int n = blockIdx.x * kWarps + (threadIdx.x >> 5); n < N; n += gridDim.x * kWarps) {
        const uint32_t *qrow = Bq + (int64_t)n * (K >> 3);
        for (int m0 = 0; m0 < M; m0 += MT) {
            float acc[MT];
#pragma unroll
            for (int i = 0; i < MT; ++i) acc[i] = 0.f;
            for (int c0 = lane; c0 < chunks; c0 += 32 * U) {
                uint4 qv[U];
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int c = c0 + 32 * u;
                    qv[u] = c < chunks ? ld_stream_v4(qrow + (int64_t)c * 4) : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int c = c0 + 32 * u;
                    if (c >= chunks) break;
                    const int g = (c * 32) / group;
                    const float s = __uint_as_float((uint32_t)S[(int64_t)n * groups + g] << 16);
                    const float z = (float)Z[(int64_t)n * groups + g];
                    const uint32_t qw[4] = {qv[u].x, qv[u].y, qv[u].z, qv[u].w};
#pragma unroll
                    for (int i = 0; i < MT; ++i) {
                        if (m0 + i >= M) break;
                        const uint16_t *arow = A + (int64_t)(m0 + i) * K + (int64_t)c * 32;
                        float sq = 0.f, sa = 0.f;
#pragma unroll
                        for (int w = 0; w < 4; ++w) {
                            const uint4 av = ld_ro_v4(arow + w * 8);
                            const uint32_t aw[4] = {av.x, av.y, av.z, av.w};
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                const float a0 = bf16lo(aw[j]), a1 = bf16hi(aw[j]);
                                const float q0 = (float)((qw[w] >> (8 * j)) & 0xFu);
                                const float q1 = (float)((qw[w] >> (8 * j + 4)) & 0xFu);
                                sq = fmaf(a0, q0, sq);
                                sq = fmaf(a1, q1, sq);
                                sa += a0 + a1;
                            }
                        }
                        acc[i] = fmaf(s, fmaf(-z, sa, sq), acc[i]);
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < MT; ++i) {
                const float v = warp_sum(acc[i]);
                if (lane == 0 && m0 + i < M) C[(int64_t)(m0 + i) * N + n] = f32_to_bf16_rn(v);
            }
        }
    }
}

// K == 0: the empty sum (plus the bias, if one is fused; silu(0) * 0 = 0).
// K == 0: the empty sum, plus the bias epilogues' bias and activation.
__global__ void k_zero_fill(uint16_t *C, int M, int N, int64_t ldc, const uint16_t *bias, int epi)
{
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < (int64_t)M * N;
         i += (int64_t)gridDim.x * blockDim.x)
        C[(i / N) * ldc + (i % N)] =
            bias ? (epi == GEMM_EPI_BIAS ? bias[i % N] : f32_to_bf16_rn(bias_act(0.f, bf16lo(bias[i % N]), epi)))
                 : (uint16_t)0;
}

template <typename Kern, typename... Args>
cudaError_t launch_pdl(Kern kern, int grid, cudaStream_t st, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(kWarps * 32, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

int rows_grid(int64_t N, int sm_count)
{
    int64_t g = (N + kWarps - 1) / kWarps;
    int64_t cap = (int64_t)sm_count * 16;
    return (int)(g < cap ? g : cap);
}

}  // namespace

cudaError_t launch_zero_fill(const GemmArgs &a, const LaunchCtx &c)
{
    int64_t total = a.M * a.N;
    int grid = (int)((total + 255) / 256);
    if (grid > c.sm_count * 8) grid = c.sm_count * 8;
    if (grid < 1) grid = 1;
    k_zero_fill<<<grid, 256, 0, c.stream>>>((uint16_t *)a.C, (int)a.M, (int)a.N, a.ldc,
                                           epi_has_bias(a.epi) ? (const uint16_t *)a.bias : nullptr, a.epi);
    return cudaGetLastError();
}

template <int EPI>
cudaError_t launch_gemv_mt(const GemmArgs &a, const Plan &p, const LaunchCtx &c, const uint16_t *A,
                           const uint16_t *B, uint16_t *C)
{
    const int M = (int)a.M, N = (int)a.N, K = (int)a.K;
    const uint16_t *bias = (const uint16_t *)a.bias;
    switch (p.m_per_pass) {
    case 1: return launch_pdl(k_gemv_bf16<1, 8, EPI>, p.grid, c.stream, A, B, C, M, N, K, a.lda, a.ldb, a.ldc, bias, a.epi);
    case 2: return launch_pdl(k_gemv_bf16<2, 8, EPI>, p.grid, c.stream, A, B, C, M, N, K, a.lda, a.ldb, a.ldc, bias, a.epi);
    case 3: return launch_pdl(k_gemv_bf16<3, 4, EPI>, p.grid, c.stream, A, B, C, M, N, K, a.lda, a.ldb, a.ldc, bias, a.epi);
    default: return launch_pdl(k_gemv_bf16<4, 4, EPI>, p.grid, c.stream, A, B, C, M, N, K, a.lda, a.ldb, a.ldc, bias, a.epi);
    }
}

cudaError_t launch_gemv_bf16(const GemmArgs &a, const Plan &p, const LaunchCtx &c)
{
    const uint16_t *A = (const uint16_t *)a.A, *B = (const uint16_t *)a.B;
    uint16_t *C = (uint16_t *)a.C;
    switch (a.epi) {
    case GEMM_EPI_BIAS:
    case GEMM_EPI_BIAS_RELU:
    case GEMM_EPI_BIAS_SILU:
    case GEMM_EPI_BIAS_GELU: return launch_gemv_mt<1>(a, p, c, A, B, C);
    case GEMM_EPI_SILU_MUL: return launch_gemv_mt<2>(a, p, c, A, B, C);
    default: return launch_gemv_mt<0>(a, p, c, A, B, C);
    }
}

cudaError_t launch_gemv_w4a16(const GemmArgs &a, const Plan &p, const LaunchCtx &c)
{
    const uint16_t *A = (const uint16_t *)a.A;
    const uint32_t *Q = (const uint32_t *)a.B;
    const uint16_t *S = (const uint16_t *)a.scales;
    const uint8_t *Z = (const uint8_t *)a.zeros;
    uint16_t *C = (uint16_t *)a.C;
    const int M = (int)a.M, N = (int)a.N, K = (int)a.K, g = (int)a.group;
    switch (p.m_per_pass) {
    case 1: return launch_pdl(k_gemv_w4a16<1>, p.grid, c.stream, A, Q, S, Z, C, M, N, K, g);
    case 2: return launch_pdl(k_gemv_w4a16<2>, p.grid, c.stream, A, Q, S, Z, C, M, N, K, g);
    default: return launch_pdl(k_gemv_w4a16<4>, p.grid, c.stream, A, Q, S, Z, C, M, N, K, g);
    }
}

int gemv_grid(int64_t N, int sm_count) { return rows_grid(N, sm_count); }

}  // namespace dbw
