// w4mma.cu -- W4A16 with the weights dequantised into registers and multiplied
// by warp-level tensor-core MMAs (mma.sync.m16n8k16, bf16 -> fp32), for
// M <= 32 tokens.
//
// The contraction is the W4A16 decode GEMM of the hk-dsl PyPI page ("Results",
// W4A16 decode GEMM (AWQ)), w[n,k] = (q[n,k] - z[n,g]) * s[n,g] with g = k / group.
// Within one quantisation group the scale and zero are constants, so
//     sum_{k in g} w[n,k] a[m,k] = s[n,g] * (D_g[n,m] - (128 + z[n,g]) * S_g[m]),
//     D_g[n,m] = sum_{k in g} (128 + q[n,k]) a[m,k],   S_g[m] = sum_{k in g} a[m,k].
// 128 + q is exact in bf16 as (0x4300 | q), so the MMA's A operand needs one
// shift and one mask per pair of weights; D_g accumulates in the MMA (fp32),
// and the zero point and scale are applied once per group in fp32.  The
// weights are never rounded to bf16 (integer-valued inputs stay exact).
//
// Work split: one CTA of eight warps per 16 weight rows; warp w takes the
// quantisation groups w, w + 8, ... over all of K and all M tokens (M/8
// rounded up MMAs of N = 8 per 16 x 16 weight block); the eight partial sums
// are added in warp order through shared memory (deterministic).  No warp
// waits on another before the final sum.
//
// Fragment mapping (thread t: groupID g = t / 4, tig = t % 4).  A group of
// `group` k is 4 * WPT packed words per row (WPT = group / 32); thread tig
// loads words WPT*tig .. WPT*tig + WPT - 1 of rows n0 + g and n0 + g + 8.  Chunk
// c (0 <= c < WPT) of the group is two 16-k MMAs over the words WPT*tig' + c of
// all four tig'.  In MMA b (0, 1) the k pair a thread holds at fragment
// positions (2 tig, 2 tig + 1) is nibble pair 2b of its word and the pair at
// (2 tig + 8, 2 tig + 9) is nibble pair 2b + 1, where nibble pair p of a word is
// the weights (p, p + 4) of its 8 k -- the two nibbles one mask extracts.  The
// activations were copied with every 8-k block in the order 0,4,1,5,2,6,3,7
// and, within a group, the block of word WPT*tig + c at position 4c + tig
// (k_w4_prep), so the B fragments of both MMAs of a chunk are one 16-byte load
// and a quad's four loads are 64 contiguous bytes.
#include <cuda_bf16.h>

#include <mutex>

#include "common.cuh"
#include "frag.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace dbw {
namespace {

constexpr int kWarpsW4 = 8;

// Activations [M, K] -> the copy in the MMA's k order, and the per-group sums
// S[g, m] (fp32, in increasing k; group-major, tokens padded to Mp with zeros,
// so a warp's sums for one group are one sector).  One thread per (token, group).
__global__ void __launch_bounds__(256) k_w4_prep(const uint16_t *__restrict__ A, uint16_t *__restrict__ Ap,
                                                 float *__restrict__ S, int M, int Mp, int K, int group)
{
    ptx::pdl_wait();                 // the workspace may still be read by the previous kernel
    ptx::pdl_launch_dependents();
    const int G = K / group;
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= Mp * G) return;
    const int m = i / G, gi = i % G;
    if (m >= M) {
        S[(int64_t)gi * Mp + m] = 0.f;
        return;
    }
    const uint4 *src = reinterpret_cast<const uint4 *>(A + (int64_t)m * K + (int64_t)gi * group);
    uint4 *dst = reinterpret_cast<uint4 *>(Ap + (int64_t)m * K + (int64_t)gi * group);
    float sum = 0.f;
    for (int b = 0; b < group / 8; ++b) {
        const uint4 a = ld_ro_v4(src + b);   // (a0 a1)(a2 a3)(a4 a5)(a6 a7)
        const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            sum += __uint_as_float(w[j] << 16);
            sum += __uint_as_float(w[j] & 0xFFFF0000u);
        }
        uint4 o;
        o.x = __byte_perm(a.x, a.z, 0x5410);   // (a0, a4)
        o.y = __byte_perm(a.x, a.z, 0x7632);   // (a1, a5)
        o.z = __byte_perm(a.y, a.w, 0x5410);   // (a2, a6)
        o.w = __byte_perm(a.y, a.w, 0x7632);   // (a3, a7)
        // block b of the group is the word thread tig = b / WPT uses in chunk
        // c = b % WPT; stored at 4 c + tig so a quad's four loads are contiguous
        const int wpt = group / 32;
        dst[4 * (b % wpt) + b / wpt] = o;
    }
    S[(int64_t)gi * Mp + m] = sum;
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void cp_async16(uint32_t smem, const void *gmem)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Per-warp ring of packed-weight groups in shared memory: 24 / WPT groups of
// 16 rows x 16 WPT bytes (6 KB per warp whatever the group size), streamed with
// cp.async so each warp keeps that many bytes of HBM requests in flight.
template <int WPT>
struct W4Ring {
    static constexpr int D = 24 / WPT;                 // groups in flight per warp
    static constexpr int SLOT = 16 * 16 * WPT;         // bytes per group: 16 rows x 4 WPT words
    static constexpr int WARP_BYTES = D * SLOT;
};

// Dynamic shared memory: the rings (reused for the final cross-warp sum), then
// the CTA's scales [16][G] (bf16) and zeros [16][G] (uint8).
template <int MT, int WPT>
constexpr int w4_ring_bytes()
{
    return kWarpsW4 * W4Ring<WPT>::WARP_BYTES > kWarpsW4 * 16 * (MT * 8 + 1) * 4
               ? kWarpsW4 * W4Ring<WPT>::WARP_BYTES
               : kWarpsW4 * 16 * (MT * 8 + 1) * 4;
}
__host__ __device__ constexpr int w4_sz_bytes(int G) { return (16 * G * 3 + 15) / 16 * 16; }
constexpr int kW4MaxGroups = kW4RegisterMaxGroups;

// MT: token groups of 8 (M <= 8 MT); WPT: group / 32.
template <int MT, int WPT>
__global__ void __launch_bounds__(kWarpsW4 * 32, MT <= 2 ? 3 : 1)
k_w4_mma(const uint16_t *__restrict__ Ap, const float *__restrict__ S, const uint32_t *__restrict__ Bq,
         const uint16_t *__restrict__ scales, const uint8_t *__restrict__ zeros, uint16_t *__restrict__ C, int M,
         int N, int K)
{
    constexpr int Mp = 8 * MT;                   // tokens of the MMAs (S is padded to it)
    using RG = W4Ring<WPT>;
    extern __shared__ __align__(16) uint8_t w4smem[];
    ptx::pdl_wait();
    ptx::pdl_launch_dependents();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, tig = lane & 3;
    const int n0 = blockIdx.x * 16;
    const int rA = n0 + g, rB = n0 + g + 8;
    const bool vA = rA < N, vB = rB < N;
    const int KW = K >> 3;                       // packed words per row
    const int G = K / (32 * WPT);                // groups
    const int ng = warp < G ? (G - warp + kWarpsW4 - 1) / kWarpsW4 : 0;   // this warp's groups
    const uint32_t ring = ptx::smem_addr(w4smem) + (uint32_t)(warp * RG::WARP_BYTES);
    // the CTA's scales and zeros, staged once (rows n0 .. n0 + 15 are contiguous in both arrays)
    uint16_t *s_sc = reinterpret_cast<uint16_t *>(w4smem + w4_ring_bytes<MT, WPT>());
    uint8_t *s_z = reinterpret_cast<uint8_t *>(s_sc + 16 * G);
    {
        const int cnt = min(16, N - n0) * G;   // valid rows only
        const uint16_t *gs = scales + (int64_t)n0 * G;
        const uint8_t *gz = zeros + (int64_t)n0 * G;
        int i0 = 0;
        if ((reinterpret_cast<uintptr_t>(gs) & 3u) == 0) {   // 4-byte pieces where aligned
            for (int i = threadIdx.x; i < cnt / 2; i += kWarpsW4 * 32)
                reinterpret_cast<uint32_t *>(s_sc)[i] = __ldg(reinterpret_cast<const uint32_t *>(gs) + i);
            i0 = cnt / 2 * 2;
        }
        for (int i = i0 + threadIdx.x; i < cnt; i += kWarpsW4 * 32) s_sc[i] = __ldg(gs + i);
        i0 = 0;
        if ((reinterpret_cast<uintptr_t>(gz) & 3u) == 0) {
            for (int i = threadIdx.x; i < cnt / 4; i += kWarpsW4 * 32)
                reinterpret_cast<uint32_t *>(s_z)[i] = __ldg(reinterpret_cast<const uint32_t *>(gz) + i);
            i0 = cnt / 4 * 4;
        }
        for (int i = i0 + threadIdx.x; i < cnt; i += kWarpsW4 * 32) s_z[i] = __ldg(gz + i);
        __syncthreads();
    }
    const uint16_t *sa = s_sc + g * G, *sb = s_sc + (g + 8) * G;
    const uint8_t *za = s_z + g * G, *zb = s_z + (g + 8) * G;

    // group j of this warp (quantisation group warp + 8 j) -> ring slot j % D
    auto issue = [&](int j) {
        if (j < ng) {
            const int gi = warp + kWarpsW4 * j;
            const uint32_t slot = ring + (uint32_t)((j % RG::D) * RG::SLOT);
            for (int i = lane; i < 16 * WPT; i += 32) {   // 16-byte pieces: row i / WPT, piece i % WPT
                const int row = i / WPT, piece = i % WPT;
                if (n0 + row < N)
                    cp_async16(slot + (uint32_t)(row * 16 * WPT + piece * 16),
                               Bq + (int64_t)(n0 + row) * KW + gi * 4 * WPT + piece * 4);
            }
        }
        cp_async_commit();   // one group per call, possibly empty, so the count stays uniform
    };
#pragma unroll 1
    for (int j = 0; j < RG::D; ++j) issue(j);

    float acc[MT][4];
#pragma unroll
    for (int h = 0; h < MT; ++h)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[h][i] = 0.f;

    // scales and zeros one group ahead
    uint32_t s_a = 0, s_b = 0, z_a = 0, z_b = 0;
    if (ng > 0) {
        s_a = vA ? sa[warp] : 0u; z_a = vA ? za[warp] : 0u;
        s_b = vB ? sb[warp] : 0u; z_b = vB ? zb[warp] : 0u;
    }
#pragma unroll 1
    for (int j = 0; j < ng; ++j) {
        const int gi = warp + kWarpsW4 * j;
        cp_async_wait<RG::D - 1>();   // this thread's copies of group j have landed
        __syncwarp();                 // ... and every lane's
        uint32_t xa[WPT], xb[WPT];
        {
            const uint32_t slot = ring + (uint32_t)((j % RG::D) * RG::SLOT) + (uint32_t)(tig * 4 * WPT);
            const uint32_t pa = slot + (uint32_t)(g * 16 * WPT), pb = slot + (uint32_t)((g + 8) * 16 * WPT);
            if constexpr (WPT == 4) {
                const uint4 u = ptx::lds128(pa), v = ptx::lds128(pb);
                xa[0] = u.x; xa[1 % WPT] = u.y; xa[2 % WPT] = u.z; xa[3 % WPT] = u.w;
                xb[0] = v.x; xb[1 % WPT] = v.y; xb[2 % WPT] = v.z; xb[3 % WPT] = v.w;
            } else {
#pragma unroll
                for (int c = 0; c < WPT; ++c) {
                    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(xa[c]) : "r"(pa + 4u * c));
                    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(xb[c]) : "r"(pb + 4u * c));
                }
            }
            if (!vA) {
#pragma unroll
                for (int c = 0; c < WPT; ++c) xa[c] = 0u;
            }
            if (!vB) {
#pragma unroll
                for (int c = 0; c < WPT; ++c) xb[c] = 0u;
            }
        }
        __syncwarp();                 // every lane has read the slot: refill it
        issue(j + RG::D);
        uint32_t t_sa = 0, t_sb = 0, t_za = 0, t_zb = 0;
        if (j + 1 < ng) {
            const int gn = gi + kWarpsW4;
            t_sa = vA ? sa[gn] : 0u; t_za = vA ? za[gn] : 0u;
            t_sb = vB ? sb[gn] : 0u; t_zb = vB ? zb[gn] : 0u;
        }
        float d[MT][4];
        // activation fragments: 16 bytes per chunk and token group, one chunk ahead
        auto load_b = [&](int c, uint4 (&bv)[MT]) {
            const int w = gi * 4 * WPT + 4 * c + tig;   // position of this thread's word in the copy
#pragma unroll
            for (int h = 0; h < MT; ++h) {
                const int tok = 8 * h + g;   // B fragment column
                bv[h] = tok < M ? ld_ro_v4(Ap + (int64_t)tok * K + 8 * w) : make_uint4(0u, 0u, 0u, 0u);
            }
        };
        uint4 bcur[MT], bnext[MT];
        load_b(0, bcur);
#pragma unroll
        for (int c = 0; c < WPT; ++c) {
            if (c + 1 < WPT) load_b(c + 1, bnext);
            // A fragments of the two MMAs of this chunk
            const uint32_t a00 = pair128(xa[c], 0), a01 = pair128(xb[c], 0), a02 = pair128(xa[c], 1),
                           a03 = pair128(xb[c], 1);
            const uint32_t a10 = pair128(xa[c], 2), a11 = pair128(xb[c], 2), a12 = pair128(xa[c], 3),
                           a13 = pair128(xb[c], 3);
#pragma unroll
            for (int h = 0; h < MT; ++h) {
                if (c == 0) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) d[h][i] = 0.f;
                }
                mma_bf16_16816(d[h], a00, a01, a02, a03, bcur[h].x, bcur[h].y);
                mma_bf16_16816(d[h], a10, a11, a12, a13, bcur[h].z, bcur[h].w);
            }
            if (c + 1 < WPT) {
#pragma unroll
                for (int h = 0; h < MT; ++h) bcur[h] = bnext[h];
            }
        }
        // per-group zero point and scale: acc += s * (D - (128 + z) * S)
        const float fsa = __uint_as_float(s_a << 16), fsb = __uint_as_float(s_b << 16);
        const float za128 = 128.f + (float)z_a, zb128 = 128.f + (float)z_b;
#pragma unroll
        for (int h = 0; h < MT; ++h) {
            const int t0 = 8 * h + 2 * tig;   // C fragment columns t0, t0 + 1
            const float2 s01 = __ldg(reinterpret_cast<const float2 *>(S + (int64_t)gi * Mp + t0));
            const float S0 = s01.x, S1 = s01.y;
            acc[h][0] = fmaf(fsa, fmaf(-za128, S0, d[h][0]), acc[h][0]);
            acc[h][1] = fmaf(fsa, fmaf(-za128, S1, d[h][1]), acc[h][1]);
            acc[h][2] = fmaf(fsb, fmaf(-zb128, S0, d[h][2]), acc[h][2]);
            acc[h][3] = fmaf(fsb, fmaf(-zb128, S1, d[h][3]), acc[h][3]);
        }
        s_a = t_sa; s_b = t_sb; z_a = t_za; z_b = t_zb;
    }
    cp_async_wait<0>();

    // the eight warps' partial sums, added in warp order (the ring's space is reused)
    __syncthreads();
    float(*red)[16][MT * 8 + 1] = reinterpret_cast<float(*)[16][MT * 8 + 1]>(w4smem);
#pragma unroll
    for (int h = 0; h < MT; ++h) {
        const int t0 = 8 * h + 2 * tig;
        red[warp][g][t0] = acc[h][0];
        red[warp][g][t0 + 1] = acc[h][1];
        red[warp][g + 8][t0] = acc[h][2];
        red[warp][g + 8][t0 + 1] = acc[h][3];
    }
    __syncthreads();
    for (int o = threadIdx.x; o < 16 * MT * 8; o += kWarpsW4 * 32) {
        const int row = o & 15, tok = o >> 4;     // neighbouring threads: neighbouring rows
        const int n = n0 + row;
        if (tok < M && n < N) {
            float v = 0.f;
#pragma unroll
            for (int w = 0; w < kWarpsW4; ++w) v += red[w][row][tok];
            C[(int64_t)tok * N + n] = f32_to_bf16_rn(v);
        }
    }
}

template <typename Kern, typename... Args>
cudaError_t launch_w4(Kern kern, int grid, int block, int smem, cudaStream_t st, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3((unsigned)block, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = st;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <int MT, int WPT>
cudaError_t launch_wpt(int grid, const LaunchCtx &c, const uint16_t *Ap, const float *S, const uint32_t *Q,
                       const uint16_t *sc, const uint8_t *zz, uint16_t *C, int M, int N, int K)
{
    const int smem = w4_ring_bytes<MT, WPT>() + w4_sz_bytes(K / (32 * WPT));
    static std::once_flag once[64];
    static cudaError_t attr_err[64];
    int dev = 0;
    cudaGetDevice(&dev);
    std::call_once(once[dev & 63], [&] {
        attr_err[dev & 63] = cudaFuncSetAttribute(k_w4_mma<MT, WPT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                  w4_ring_bytes<MT, WPT>() + w4_sz_bytes(kW4MaxGroups));
    });
    if (attr_err[dev & 63] != cudaSuccess) return attr_err[dev & 63];
    return launch_w4(k_w4_mma<MT, WPT>, grid, kWarpsW4 * 32, smem, c.stream, Ap, S, Q, sc, zz, C, M, N, K);
}

template <int MT>
cudaError_t launch_mt(const GemmArgs &a, const LaunchCtx &c, const uint16_t *Ap, const float *S, int grid)
{
    const uint32_t *Q = (const uint32_t *)a.B;
    const uint16_t *sc = (const uint16_t *)a.scales;
    const uint8_t *zz = (const uint8_t *)a.zeros;
    uint16_t *C = (uint16_t *)a.C;
    const int M = (int)a.M, N = (int)a.N, K = (int)a.K;
    switch (a.group) {
    case 32: return launch_wpt<MT, 1>(grid, c, Ap, S, Q, sc, zz, C, M, N, K);
    case 64: return launch_wpt<MT, 2>(grid, c, Ap, S, Q, sc, zz, C, M, N, K);
    default: return launch_wpt<MT, 4>(grid, c, Ap, S, Q, sc, zz, C, M, N, K);
    }
}

}  // namespace

int w4_register_grid(int64_t N) { return (int)((N + 15) / 16); }

cudaError_t launch_w4_register(const GemmArgs &a, const Plan &p, const LaunchCtx &c)
{
    if (!c.act_copy) return cudaErrorInvalidValue;
    uint16_t *Ap = (uint16_t *)c.act_copy;
    float *S = reinterpret_cast<float *>(Ap + (a.M * a.K + 127) / 128 * 128);   // after the copy, 256-B aligned
    const int M = (int)a.M, K = (int)a.K, grp = (int)a.group;
    const int Mp = 8 * p.m_per_pass;
    const int items = Mp * (K / grp);
    cudaError_t e =
        launch_w4(k_w4_prep, (items + 255) / 256, 256, 0, c.stream, (const uint16_t *)a.A, Ap, S, M, Mp, K, grp);
    if (e != cudaSuccess) return e;
    switch (p.m_per_pass) {
    case 1: return launch_mt<1>(a, c, Ap, S, p.grid);
    case 2: return launch_mt<2>(a, c, Ap, S, p.grid);
    default: return launch_mt<4>(a, c, Ap, S, p.grid);
    }
}

}  // namespace dbw
