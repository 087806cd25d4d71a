// w4gemv.cu -- W4A16 for up to 16 tokens: the weights stream through per-warp
// TMA rings and are dequantised into the A fragments of warp-level MMAs
// (mma.sync.m16n8k16, bf16 -> fp32; weight rows on the MMA's M side, tokens
// on its N side), with the K dimension shared out over every warp of the
// device.
//
// The contraction is the W4A16 decode GEMM of the hk-dsl PyPI page ("Results",
// W4A16 decode GEMM (AWQ)): w[n,k] = (q[n,k] - z[n,g]) * s[n,g], g = k / group.
// Within one quantisation group the scale and zero are constants, so
//     sum_{k in g} w a = s * (D_g - (128 + z) S_g),
//     D_g = sum_{k in g} (128 + q) a,         S_g = sum_{k in g} a.
// 128 + q is exact in bf16 as (0x4300 | q); D_g accumulates in fp32 in the
// MMA, and so does S_g, from an A operand of ones (bf16 1.0) against the same
// activation operands: every row of that accumulator holds the token's group
// sum.  One multiply-add by the (exact) factor -(128 + z) and one by s per
// output close the group.  The weights are never rounded to bf16.
//
// Work split (a decode GEMM moves a few tens of MB: the weights of each SM
// must all be in flight at once, and no warp may carry a long serial chain).
// A cluster of two CTAs of four warps takes a tile of 32 weight rows over
// all of K; its eight warps take equal runs of the 128-k chunks.  Before the
// grid dependency wait each warp asks L2 for its chunks and the CTA for its
// scale and zero rows (prefetches only: nothing is consumed before the wait);
// after it a warp streams its chunks by TMA into a ring of its own (one 2-D
// box of 16 words x 32 rows, 64-byte swizzle, one mbarrier per slot; five
// slots) and refills a slot as soon as it has read it, and the tile's scale
// and zero rows (contiguous in memory) arrive by two bulk copies.  A group's
// activation words are loaded (straight from A) while the previous group is
// multiplied.  The eight partial sums meet in shared memory, each CTA adding
// its four in warp order and the second handing its sum to the first through
// distributed shared memory (deterministic).  Three CTAs per SM: half tiles
// keep the SMs' shares of the work even when the tiles are not a multiple of
// the SM count (224 whole tiles on 152 SMs would give some SMs two and others
// one; 448 halves give every SM two or three).
//
// Fragment mapping (lane: g = lane / 4, t = lane % 4).  MMA row m of block b
// is tile row 16 b + m.  Within a group a row has 4 WPT words (WPT = group /
// 32); lane t holds words WPT t .. WPT t + WPT - 1 of rows g and g + 8, and
// its word i feeds two k-steps: nibble pairs (0,4) and (1,5) at the
// fragment's k positions (2t, 2t+1) and (2t+8, 2t+9), then pairs (2,6) and
// (3,7).  The lane's 16-byte activation word (the same 8 k) is permuted to
// the order 0,4,1,5,2,6,3,7 in registers (four byte permutes), so it gives
// the B operands of both k-steps.  With 64-byte rows and the 64-byte swizzle
// the eight rows a quarter-warp reads fall on distinct bank groups.
#include <cuda.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "frag.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "waits.cuh"

namespace dbw {
namespace {

constexpr int kRows = kW4GemvRows;               // weight rows per tile (two blocks of sixteen)
constexpr int kWarps = kW4GemvWarps;
constexpr int kSlots = 5;                        // ring slots per warp
constexpr int kSlot = kRows * 64;                // one 128-k chunk: 32 rows x 16 words
constexpr int kRing = kWarps * kSlots * kSlot;   // 40 KB
constexpr int kMaxGroups = kW4GemvMaxGroups;     // scale and zero rows staged whole
constexpr int kSzOff = kRing;                    // scales [32][G] bf16, zeros [32][G] u8
constexpr int kBarOff = kSzOff + kRows * kMaxGroups * 3;
constexpr int kRedOff = kBarOff + kWarps * kSlots * 8;   // the partner CTA's sum [32][16] fp32
constexpr int kPartOff = kRedOff + kRows * 16 * 4;      // the warps' sums [warp][32][16] fp32
constexpr int kSzBar = kPartOff + kWarps * kRows * 16 * 4;
constexpr int kFlagOff = kSzBar + 8;
constexpr int kSmem = kFlagOff + 8 + 1024;       // + alignment slack

// Words i of rows r and r + 8 of group h for lane t, from a slot (64-byte
// rows, 16-byte piece c of row r at piece c ^ ((r / 2) % 4)).
template <int WPT>
__device__ __forceinline__ void load_words(uint32_t slot, int r, int h, int t, uint32_t (&xa)[WPT],
                                           uint32_t (&xb)[WPT])
{
    const int lb = h * (16 * WPT) + 4 * WPT * t;   // logical byte of the lane's first word in the row
    const uint32_t off = (uint32_t)(((((lb >> 4) ^ ((r >> 1) & 3)) << 4)) | (lb & 15));
    const uint32_t pa = slot + (uint32_t)(r * 64) + off, pb = pa + 8u * 64u;   // rows r, r + 8: same swizzle
    if constexpr (WPT == 4) {
        const uint4 v = ptx::lds128(pa), w = ptx::lds128(pb);
        xa[0] = v.x;
        xa[1 % WPT] = v.y;
        xa[2 % WPT] = v.z;
        xa[3 % WPT] = v.w;
        xb[0] = w.x;
        xb[1 % WPT] = w.y;
        xb[2 % WPT] = w.z;
        xb[3 % WPT] = w.w;
    } else if constexpr (WPT == 2) {
        asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(xa[0]), "=r"(xa[1 % WPT]) : "r"(pa));
        asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(xb[0]), "=r"(xb[1 % WPT]) : "r"(pb));
    } else {
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(xa[0]) : "r"(pa));
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(xb[0]) : "r"(pb));
    }
}

// Activation operands of one group: the lane's 16-byte activation words of
// token 8u + g, as loaded (k order 0..7; permuted when used).
template <int NT, int WPT>
struct GroupAct {
    uint4 a[NT][WPT];
};

template <int NT, int WPT>
__global__ void __launch_bounds__(kWarps * 32, 3)
k_w4_gemv(const __grid_constant__ CUtensorMap tmQ, const uint16_t *__restrict__ A, const uint16_t *__restrict__ scales,
          const uint8_t *__restrict__ zeros, uint16_t *__restrict__ C, int M, int N, int K, int *__restrict__ d_error,
          int stall)
{
    constexpr int GROUP = 32 * WPT;
    constexpr int GU = 4 / WPT;   // groups per 128-k chunk
    constexpr int TP = 8 * NT;    // tokens of the MMAs
    extern __shared__ uint8_t gv_raw[];
    uint8_t *smem = gv_raw + ((1024u - (ptx::smem_addr(gv_raw) & 1023u)) & 1023u);
    const uint32_t sbase = ptx::smem_addr(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    // a cluster of two CTAs per tile, each taking half of K
    const uint32_t rank = ptx::cluster_ctarank();
    const int tile = blockIdx.x >> 1, n0 = tile * kRows;
    const int G = K / GROUP;
    const int nk = (K + 127) >> 7;                                    // 128-k chunks
    const int wk = (int)rank * kWarps + warp;                         // this warp among the tile's eight
    const int c0 = wk * nk / (2 * kWarps), nu = (wk + 1) * nk / (2 * kWarps) - c0;   // its chunks
    const uint32_t ring = sbase + (uint32_t)(warp * kSlots * kSlot);
    const uint32_t bar0 = sbase + (uint32_t)(kBarOff + warp * kSlots * 8);
    const uint32_t szbar = sbase + (uint32_t)kSzBar;
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + kFlagOff);
    // the tile's scales [32][G] (bf16) and zeros [32][G] (u8), rows beyond N zero
    const uint16_t *sS = reinterpret_cast<const uint16_t *>(smem + kSzOff);
    const uint8_t *sZ = smem + kSzOff + kRows * G * 2;
    const uint64_t policy = ptx::policy_evict_first();
    const int vr = min(kRows, N - n0);   // rows of the tile within N
    // the scale and zero rows of a tile are contiguous: two bulk copies when
    // their sizes are whole 16-byte units, else plain loads
    const bool bulk = (vr * G) % 16 == 0;

    // chunk c0 + q of this warp -> slot q % kSlots (lane 0 only)
    auto issue = [&](int q) {
        const uint32_t bar = bar0 + 8u * (uint32_t)(q % kSlots);
        ptx::mbar_arrive_expect_tx(bar, (uint32_t)kSlot);
        ptx::tma_load_2d(ring + (uint32_t)((q % kSlots) * kSlot), &tmQ, bar, (c0 + q) * 16, n0, policy);
    };
    // the tile's scale and zero rows into shared memory (thread 0 issues the
    // copies; every thread takes part in the plain loads)
    auto load_sz = [&]() {
        if (bulk && threadIdx.x == 0 && !stall) {
            ptx::mbar_arrive_expect_tx(szbar, (uint32_t)(vr * G * 3));
            bulk_load(sbase + (uint32_t)kSzOff, scales + (int64_t)n0 * G, (uint32_t)(vr * G * 2), szbar);
            bulk_load(sbase + (uint32_t)(kSzOff + kRows * G * 2), zeros + (int64_t)n0 * G, (uint32_t)(vr * G), szbar);
        }
        uint16_t *wS = reinterpret_cast<uint16_t *>(smem + kSzOff);
        uint8_t *wZ = smem + kSzOff + kRows * G * 2;
        for (int i = (bulk && !stall ? vr * G : 0) + threadIdx.x; i < kRows * G; i += kWarps * 32) {
            const bool v = i < vr * G;
            wS[i] = v ? scales[(int64_t)n0 * G + i] : (uint16_t)0;
            wZ[i] = v ? zeros[(int64_t)n0 * G + i] : (uint8_t)0;
        }
    };

    // Before the grid dependency wait only L2 prefetches of this CTA's
    // weights and scale rows are issued (L2 is the coherence point, so
    // nothing stale is consumed); the copies into shared memory follow it.
    if (threadIdx.x == 0) {
        *abort_flag = 0u;
        ptx::mbar_init(szbar, 1);
        if (bulk) {
            bulk_prefetch_l2(scales + (int64_t)n0 * G, (uint32_t)(vr * G * 2));
            bulk_prefetch_l2(zeros + (int64_t)n0 * G, (uint32_t)(vr * G));
        }
    }
    if (lane == 0) {
        for (int s = 0; s < kSlots; ++s) ptx::mbar_init(bar0 + 8u * (uint32_t)s, 1);
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tmQ);
        for (int q = 0; q < nu; ++q) ptx::tma_prefetch_l2_2d(&tmQ, (c0 + q) * 16, n0);
    }
    __syncthreads();   // barriers and the abort flag initialised
    ptx::pdl_wait();   // the activations (and C) may belong to the previous kernel
    ptx::pdl_launch_dependents();
    int issued = 0;
    if (lane == 0 && !stall)
        for (; issued < kSlots && issued < nu; ++issued) issue(issued);

    // lanes of absent tokens (8u + g >= M) read token M - 1's row: their MMA
    // columns are never stored
    const uint16_t *arow[NT];
#pragma unroll
    for (int u = 0; u < NT; ++u) arow[u] = A + (int64_t)min(8 * u + g, M - 1) * K + 8 * WPT * t;
    auto load_act = [&](int gi, GroupAct<NT, WPT> &o) {
#pragma unroll
        for (int u = 0; u < NT; ++u)
#pragma unroll
            for (int i = 0; i < WPT; ++i) o.a[u][i] = ld_ro_v4(arow[u] + gi * GROUP + 8 * i);
    };

    const int gbeg = c0 * GU, gend = min(G, (c0 + nu) * GU);   // this warp's groups
    float acc[2][NT][4];
    int q = 0;   // chunks of the sequence consumed
    // group gi of the current tile with its activations in `cur`, fetching
    // the next group's into `nxt`
    auto step = [&](int gi, const GroupAct<NT, WPT> &cur, GroupAct<NT, WPT> &nxt) {
        const int h = gi % GU;
        const uint32_t slot = ring + (uint32_t)((q % kSlots) * kSlot);
        if (gi + 1 < gend) load_act(gi + 1, nxt);
        if (h == 0 && !wait_bar_warp(bar0 + 8u * (uint32_t)(q % kSlots), (uint32_t)(q / kSlots) & 1u, abort_flag,
                                     d_error))
            return;
        // rows g + 8e: the scale and -(128 + z) = (2^23 - 128) - (2^23 + z);
        // lane t of a quad reads row g + 8t, the quad shares them
        const float s_t = __uint_as_float((uint32_t)sS[(g + 8 * t) * G + gi] << 16);
        const float cz_t = 8388480.f - __uint_as_float(0x4B000000u | (uint32_t)sZ[(g + 8 * t) * G + gi]);
        float s[4], cz[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            s[e] = __shfl_sync(0xffffffffu, s_t, (lane & ~3) | e);
            cz[e] = __shfl_sync(0xffffffffu, cz_t, (lane & ~3) | e);
        }
        uint32_t xa[2][WPT], xb[2][WPT];
#pragma unroll
        for (int b = 0; b < 2; ++b) load_words<WPT>(slot, 16 * b + g, h, t, xa[b], xb[b]);
        // D_g per (block, token tile), for one token tile in two chains (the
        // k-steps of a word alternate between them; two token tiles already
        // give four), and S_g per token tile from an A operand of ones: every
        // accumulator row then holds the token's group sum
        constexpr uint32_t ONES = 0x3F803F80u;
        constexpr int NCH = NT == 1 ? 2 : 1;
        float d[2][NT][NCH][4], sg[NT][4];
#pragma unroll
        for (int u = 0; u < NT; ++u)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                sg[u][e] = 0.f;
#pragma unroll
                for (int b = 0; b < 2; ++b)
#pragma unroll
                    for (int c = 0; c < NCH; ++c) d[b][u][c][e] = 0.f;
            }
#pragma unroll
        for (int i = 0; i < WPT; ++i) {
            // B operands: the word's 8-k block in the order 0,4,1,5,2,6,3,7, so
            // that bf16 pair j of an A register (nibbles p, p + 4) meets (a_p, a_{p+4})
            uint32_t bo[NT][4];
#pragma unroll
            for (int u = 0; u < NT; ++u) {
                const uint4 r = cur.a[u][i];
                bo[u][0] = __byte_perm(r.x, r.z, 0x5410);   // (a0, a4)
                bo[u][1] = __byte_perm(r.x, r.z, 0x7632);   // (a1, a5)
                bo[u][2] = __byte_perm(r.y, r.w, 0x5410);   // (a2, a6)
                bo[u][3] = __byte_perm(r.y, r.w, 0x7632);   // (a3, a7)
                mma_acc(sg[u], ONES, ONES, ONES, ONES, bo[u][0], bo[u][1]);
                mma_acc(sg[u], ONES, ONES, ONES, ONES, bo[u][2], bo[u][3]);
            }
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                const uint32_t a00 = pair128(xa[b][i], 0), a01 = pair128(xb[b][i], 0),
                               a02 = pair128(xa[b][i], 1), a03 = pair128(xb[b][i], 1);
                const uint32_t a10 = pair128(xa[b][i], 2), a11 = pair128(xb[b][i], 2),
                               a12 = pair128(xa[b][i], 3), a13 = pair128(xb[b][i], 3);
#pragma unroll
                for (int u = 0; u < NT; ++u) {
                    mma_acc(d[b][u][0], a00, a01, a02, a03, bo[u][0], bo[u][1]);
                    mma_acc(d[b][u][NCH - 1], a10, a11, a12, a13, bo[u][2], bo[u][3]);
                }
            }
        }
        // acc += s (D_g - (128 + z) S_g)
#pragma unroll
        for (int b = 0; b < 2; ++b)
#pragma unroll
            for (int u = 0; u < NT; ++u)
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    acc[b][u][e] = fmaf(s[2 * b + (e >> 1)],
                                        fmaf(cz[2 * b + (e >> 1)], sg[u][e],
                                             NCH == 1 ? d[b][u][0][e] : d[b][u][0][e] + d[b][u][NCH - 1][e]),
                                        acc[b][u][e]);
        if (h == GU - 1 || gi + 1 == gend) {
            // every lane's reads of the slot have completed (their values were
            // used above): hand it back to the copy engine for chunk q + slots
            __syncwarp();
            if (lane == 0 && !stall && issued < nu && !*abort_flag) {
                ptx::fence_proxy_async_smem();
                issue(issued++);
            }
            ++q;
        }
    };

    GroupAct<NT, WPT> A0, A1;
    if (gbeg < gend) load_act(gbeg, A0);
    load_sz();
    __syncthreads();   // the plain-loaded scale rows
    if (bulk && !stall) {
        // (a copy issued before an abort still lands before the CTA leaves)
        if (!wait_bar(szbar, 0u, abort_flag, d_error) && threadIdx.x == 0) wait_bar_drain(szbar, 0u);
    }
    __syncwarp();
#pragma unroll
    for (int b = 0; b < 2; ++b)
#pragma unroll
        for (int u = 0; u < NT; ++u)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[b][u][e] = 0.f;
    // the warp's groups, two per pass (activations alternate between A0 and A1)
#pragma unroll 1
    for (int gi = gbeg; gi < gend && !*abort_flag; gi += 2) {
        step(gi, A0, A1);
        if (gi + 1 < gend) step(gi + 1, A1, A0);
    }
    // the eight warps' sums of the tile [row][token]: each CTA adds its four
    // in warp order, the second CTA hands its sum to the first through
    // distributed shared memory, and the first adds the two (deterministic)
    // and stores
    float *part = reinterpret_cast<float *>(smem + kPartOff);   // [warp][row][token]
    float *mine = part + warp * (kRows * TP);
#pragma unroll
    for (int b = 0; b < 2; ++b)
#pragma unroll
        for (int u = 0; u < NT; ++u)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                mine[(16 * b + g + 8 * (e >> 1)) * TP + 8 * u + 2 * t + (e & 1)] = acc[b][u][e];
    __syncthreads();
    float *red = reinterpret_cast<float *>(smem + kRedOff);   // the partner's sum (in the first CTA)
    float v[(kRows * TP + kWarps * 32 - 1) / (kWarps * 32)];
#pragma unroll
    for (int r = 0; r < (int)(sizeof(v) / sizeof(float)); ++r) {
        const int i = threadIdx.x + r * kWarps * 32;
        v[r] = 0.f;
        if (i < kRows * TP) {
#pragma unroll
            for (int w = 0; w < kWarps; ++w) v[r] += part[w * (kRows * TP) + i];
            if (rank == 1) {
                const uint32_t dst = ptx::map_cluster(ptx::smem_addr(red + i), 0u);
                asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(dst), "f"(v[r]) : "memory");
            }
        }
    }
    ptx::cluster_arrive_release();
    ptx::cluster_wait();
    if (rank == 0 && !*abort_flag) {
#pragma unroll
        for (int r = 0; r < (int)(sizeof(v) / sizeof(float)); ++r) {
            const int i = threadIdx.x + r * kWarps * 32;
            const int row = i / TP, tok = i % TP;
            if (i < kRows * TP && tok < M && n0 + row < N)
                C[(int64_t)tok * N + n0 + row] = f32_to_bf16_rn(v[r] + red[i]);
        }
    }
    if (*abort_flag && lane == 0 && !stall) {
        // chunks issued but not consumed land before the ring is released
        for (int q2 = q; q2 < issued; ++q2)
            wait_bar_drain(bar0 + 8u * (uint32_t)(q2 % kSlots), (uint32_t)(q2 / kSlots) & 1u);
    }
}

template <int NT, int WPT>
cudaError_t launch_t(const CUtensorMap &m, const GemmArgs &a, const LaunchCtx &c, int grid)
{
    auto kern = k_w4_gemv<NT, WPT>;
    static std::once_flag once[64];
    static cudaError_t attr_err[64];
    int dev = 0;
    cudaGetDevice(&dev);
    std::call_once(once[dev & 63], [&] {
        attr_err[dev & 63] = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    });
    if (attr_err[dev & 63] != cudaSuccess) return attr_err[dev & 63];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(kWarps * 32, 1, 1);
    cfg.dynamicSmemBytes = kSmem;
    cfg.stream = c.stream;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    at[1].id = cudaLaunchAttributeClusterDimension;
    at[1].val.clusterDim.x = 2;
    at[1].val.clusterDim.y = 1;
    at[1].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, m, (const uint16_t *)a.A, (const uint16_t *)a.scales,
                              (const uint8_t *)a.zeros, (uint16_t *)a.C, (int)a.M, (int)a.N, (int)a.K, c.d_error,
                              g_debug_stall);
}

template <int NT>
cudaError_t launch_nt(const CUtensorMap &m, const GemmArgs &a, const LaunchCtx &c, int grid)
{
    switch (a.group) {
    case 32: return launch_t<NT, 1>(m, a, c, grid);
    case 64: return launch_t<NT, 2>(m, a, c, grid);
    default: return launch_t<NT, 4>(m, a, c, grid);
    }
}

}  // namespace

// A cluster of two CTAs per 32-row tile (the planner takes this kernel when
// they are all resident at once, three CTAs per SM).
int w4_gemv_grid(int64_t N) { return (int)(2 * ((N + kRows - 1) / kRows)); }

cudaError_t launch_w4_gemv(const GemmArgs &a, const Plan &p, const LaunchCtx &c)
{
    CUtensorMap m;
    if (!make_map_words16(&m, a.B, a.N, a.K, kRows)) return cudaErrorInvalidValue;
    return p.tile_m <= 8 ? launch_nt<1>(m, a, c, p.grid) : launch_nt<2>(m, a, c, p.grid);
}

}  // namespace dbw
