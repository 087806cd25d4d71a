// w4band.cu -- W4A16 decode for up to 8 tokens on bands of weight rows: the
// band structure of the bf16 band kernel (gemvband.cu) with the W4A16
// arithmetic of the fragment kernels (w4gemv.cu).
//
// The contraction is the W4A16 decode GEMM of the hk-dsl PyPI page ("Results",
// W4A16 decode GEMM (AWQ)): w[n,k] = (q[n,k] - z[n,g]) * s[n,g], g = k / group.
// Within one quantisation group the scale and zero are constants, so
//     sum_{k in g} w a = s * (D_g - (128 + z) S_g),
//     D_g = sum_{k in g} (128 + q) a,         S_g = sum_{k in g} a,
// with 128 + q exact in bf16 as (0x4300 | q); D_g and S_g (from an A operand
// of bf16 ones) accumulate in fp32 in warp-level MMAs (mma.sync.m16n8k16,
// weight rows on the MMA's M side, tokens on its N side), and one multiply-add
// by -(128 + z) (exact) and one by s per output close the group.  The
// weights are never rounded to bf16, so integer cases are exact.
//
// Work split: CTA c of G takes weight rows [c N / G, (c + 1) N / G) (at most
// 64) over all of K, so no partial sum leaves the SM.  A stage is a k-chunk of
// the band: 256-k TMA boxes (32 packed words = 128 bytes per row, 128-byte
// swizzle) of 16 * ceil(rows / 16) rows from the band's first row, fetched by
// one 3-D copy when K is a multiple of 256 (the rows past the band belong to
// the neighbouring band, which asks for them at the same time; their sums are
// dropped).  A band that fits the shared-memory budget whole is requested at
// once in four stages, one per set of MMA warps; a longer one streams through
// eight slots, two owned by each set (the previous use of a slot is always
// the same set's previous stage, so no parity wait can see a phase two steps
// away); the three MMA warps of a set take every third quantisation group of
// their stages.  The band's scale and zero rows (contiguous in memory) are staged in
// shared memory once, after the grid dependency wait; before it the copy
// warp only asks L2 for the first stages.  The activations come straight from
// A (16 bytes per lane and packed word, through L1), permuted in registers to
// the nibble-pair order.  The twelve MMA warps (three per SM sub-partition,
// at most 128 registers a thread) keep their own sums; they meet once in
// shared memory, added in warp order (deterministic).
//
// Fragment mapping (lane: g = lane / 4, t = lane % 4), as in w4gemv.cu: a
// group has 4 WPT words per row (WPT = group / 32); lane t holds words
// WPT t .. WPT t + WPT - 1 of rows g and g + 8 of each 16-row MMA tile, and its
// word i feeds two k-steps: nibble pairs (0,4) and (1,5) at the fragment's k
// positions (2t, 2t+1) and (2t+8, 2t+9), then pairs (2,6) and (3,7); the
// lane's 16-byte activation word (the same 8 k) is permuted to the order
// 0,4,1,5,2,6,3,7 (four byte permutes).
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

constexpr int kMmaWarps = 12;                     // three per stage: a set takes every fourth stage
constexpr int kPairs = 4;                         // consumer sets
constexpr int kPer = kMmaWarps / kPairs;          // warps per set
constexpr int kThreads = (kMmaWarps + 1) * 32;   // + the copy warp
constexpr int kMaxTiles = kW4BandMaxRows / 16;    // 16-row MMA tiles per band
constexpr int kMaxStages = 8;
constexpr int kSmemCap = 200 * 1024;
constexpr int kBoxK = 256;                        // k per box row: 32 packed words, 128 bytes

struct W4BandGeo {
    int nkb;           // 256-k boxes per stage
    int stages;        // ring slots: 4 (the whole band at once, one stage per MMA warp) or 8
    int wrows;         // weight rows per box: 16 * tiles
    int tiles;
    int stage_bytes;   // nkb * wrows * 128
    int sz_bytes;      // staged scales [wrows][G] (bf16) and zeros [wrows][G] (u8), 16-byte multiple
};

constexpr int red_bytes(int nt) { return kMmaWarps * 16 * kMaxTiles * 8 * nt * 4; }
constexpr int kBarBytes = 8 * (2 * kMaxStages + 2) + 8;

int w4band_nt(int64_t M) { return M <= 8 ? 1 : 2; }   // (M <= kW4BandMaxTokens = 8: one token tile)

int w4band_smem(const W4BandGeo &g, int nt)
{
    return g.stages * g.stage_bytes + g.sz_bytes + red_bytes(nt) + kBarBytes + 1024;   // + alignment slack
}

// Words i = 0..WPT-1 of lane t in group h of a box row r (128-byte rows,
// 16-byte piece c of row r at piece c ^ (r % 8)).
template <int WPT>
__device__ __forceinline__ void load_words(uint32_t row_addr, int sw, int h, int t, uint32_t (&x)[WPT])
{
    const int lb = h * (16 * WPT) + 4 * WPT * t;   // logical byte of the lane's first word
    const uint32_t pa = row_addr + (uint32_t)((((lb >> 4) ^ sw) << 4) | (lb & 15));
    if constexpr (WPT == 4) {
        const uint4 v = ptx::lds128(pa);
        x[0] = v.x;
        x[1 % WPT] = v.y;
        x[2 % WPT] = v.z;
        x[3 % WPT] = v.w;
    } else if constexpr (WPT == 2) {
        asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(x[0]), "=r"(x[1 % WPT]) : "r"(pa));
    } else {
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(x[0]) : "r"(pa));
    }
}

template <int NT, int WPT>
__global__ void __launch_bounds__(kThreads, 1)
k_w4_band(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmQ3, int three_d,
          const uint16_t *__restrict__ A, const uint16_t *__restrict__ scales, const uint8_t *__restrict__ zeros,
          uint16_t *__restrict__ C, int M, int N, int K, W4BandGeo geo, int *__restrict__ d_error, int stall)
{
    constexpr int GROUP = 32 * WPT;
    constexpr int GU = kBoxK / GROUP;   // groups per box
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (sbase - raw);
    const int ring = geo.stages * geo.stage_bytes;
    uint16_t *sS = reinterpret_cast<uint16_t *>(smem + ring);
    const int G = K / GROUP;
    uint8_t *sZ = smem + ring + geo.wrows * G * 2;
    float *red = reinterpret_cast<float *>(smem + ring + geo.sz_bytes);
    const uint32_t bars = sbase + (uint32_t)(ring + geo.sz_bytes + red_bytes(NT));
    auto FULL = [&](int s) { return bars + 8u * (uint32_t)s; };
    auto EMPTY = [&](int s) { return bars + 8u * (uint32_t)(kMaxStages + s); };
    const uint32_t SZB = bars + 8u * (2 * kMaxStages);
    const uint32_t REDB = SZB + 8u;
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + ring + geo.sz_bytes +
                                                                          red_bytes(NT) + 8 * (2 * kMaxStages + 2));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r0 = (int)((int64_t)blockIdx.x * N / gridDim.x);
    const int rows = (int)((int64_t)(blockIdx.x + 1) * N / gridDim.x - r0);
    const int kbs = (K + kBoxK - 1) / kBoxK;             // 256-k boxes over K
    const int nch = (kbs + geo.nkb - 1) / geo.nkb;       // stages over K
    const uint32_t wbox = (uint32_t)geo.wrows * 128u;
    // ring slot of stage ch: MMA warps w and w + 4 consume the stages
    // ch = w mod 4 (alternate groups each) and own slots w and w + 4 (with
    // four slots, slot w)
    auto slot = [&](int ch) { return geo.stages >= 4 ? (ch & 3) + 4 * ((ch >> 2) % (geo.stages >> 2)) : ch; };

    if (threadIdx.x == 0) {
        for (int s = 0; s < geo.stages; ++s) {
            ptx::mbar_init(FULL(s), 1);
            ptx::mbar_init(EMPTY(s), kPer);   // the set of MMA warps that consumes it
        }
        ptx::mbar_init(SZB, kMmaWarps);
        ptx::mbar_init(REDB, kMmaWarps);
        *abort_flag = 0u;
        ptx::fence_mbar_init();
    }
    __syncthreads();

    if (warp == kMmaWarps) {
        // ---------------------------------------------------------------- copy warp
        if (lane == 0) {
            ptx::prefetch_tmap(three_d ? &tmQ3 : &tmQ);
            if (three_d) {
                for (int ch = 0; ch < std::min(nch, geo.stages); ++ch)
                    ptx::tma_prefetch_l2_3d(&tmQ3, 0, r0, ch * geo.nkb);
            } else {
                for (int b = 0; b < std::min(kbs, geo.stages * geo.nkb); ++b)
                    ptx::tma_prefetch_l2_2d(&tmQ, 32 * b, r0);
            }
        }
        ptx::pdl_wait();
        ptx::pdl_launch_dependents();
        const uint64_t pol = ptx::policy_evict_first();
        int issued = 0;
        if (!stall) {
            for (int ch = 0; ch < nch; ++ch) {
                const int s = slot(ch);
                if (ch >= geo.stages && !wait_bar_warp(EMPTY(s), (uint32_t)((ch / geo.stages - 1) & 1), abort_flag,
                                                       d_error))
                    break;
                if (lane == 0) {
                    const int b0 = ch * geo.nkb, nb = std::min(geo.nkb, kbs - b0);
                    const uint32_t st = sbase + (uint32_t)(s * geo.stage_bytes);
                    if (three_d) {
                        ptx::mbar_arrive_expect_tx(FULL(s), (uint32_t)geo.nkb * wbox);   // past K: zeros
                        ptx::tma_load_3d(st, &tmQ3, FULL(s), 0, r0, b0, pol);
                    } else {
                        ptx::mbar_arrive_expect_tx(FULL(s), (uint32_t)nb * wbox);
                        for (int b = 0; b < nb; ++b)
                            ptx::tma_load_2d(st + (uint32_t)b * wbox, &tmQ, FULL(s), 32 * (b0 + b), r0, pol);
                    }
                }
                __syncwarp();
                ++issued;
            }
        }
        if (lane == 0)
            for (int ch = std::max(0, issued - geo.stages); ch < issued; ++ch)
                wait_bar_drain(FULL(slot(ch)), (uint32_t)((ch / geo.stages) & 1));
        return;
    }

    // -------------------------------------------------------------------- MMA warps
    ptx::pdl_wait();   // the activations (and C) may belong to the previous kernel
    // the band's scale and zero rows (contiguous: rows r0.. of [N][G]); rows
    // of the last tile past the band read as zero
    for (int i = threadIdx.x; i < geo.wrows * G; i += kMmaWarps * 32) {
        const bool v = i < rows * G;
        sS[i] = v ? scales[(int64_t)r0 * G + i] : (uint16_t)0;
        sZ[i] = v ? zeros[(int64_t)r0 * G + i] : (uint8_t)0;
    }
    uint32_t szphase = 0;
    bool ok = group_sync_warp(SZB, szphase, abort_flag, d_error);

    const int g = lane >> 2, t = lane & 3;
    const int tiles = (rows + 15) >> 4;   // this band's MMA tiles (<= geo.tiles)
    // lanes of absent tokens (8u + g >= M) read token M - 1's row: their MMA
    // columns are never stored
    const uint16_t *arow[NT];
#pragma unroll
    for (int u = 0; u < NT; ++u) arow[u] = A + (int64_t)min(8 * u + g, M - 1) * K + 8 * WPT * t;
    float acc[kMaxTiles][NT][4];
#pragma unroll
    for (int i = 0; i < kMaxTiles; ++i)
#pragma unroll
        for (int u = 0; u < NT; ++u)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[i][u][e] = 0.f;
    constexpr uint32_t ONES = 0x3F803F80u;
    constexpr int NCH = 1;   // D_g chains per token tile (the tiles give independent chains)

    // a group's activation words (16 bytes per token tile and packed word)
    auto load_act = [&](int gi, uint4 (&av)[NT][WPT]) {
#pragma unroll
        for (int u = 0; u < NT; ++u)
#pragma unroll
            for (int i = 0; i < WPT; ++i) av[u][i] = ld_ro_v4(arow[u] + (int64_t)gi * GROUP + 8 * i);
    };
    // group gi of the box at `wb` (group h within it), its activations in av
    auto group = [&](uint32_t wb, int h, int gi, const uint4 (&av)[NT][WPT]) {
        float d[kMaxTiles][NT][NCH][4], sg[NT][2][4];   // S_g in two chains
#pragma unroll
        for (int u = 0; u < NT; ++u)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                sg[u][0][e] = sg[u][1][e] = 0.f;
#pragma unroll
                for (int mt = 0; mt < kMaxTiles; ++mt)
#pragma unroll
                    for (int c = 0; c < NCH; ++c) d[mt][u][c][e] = 0.f;
            }
        uint32_t xa[kMaxTiles][WPT], xb[kMaxTiles][WPT];   // words of rows g and g + 8 of each tile
#pragma unroll
        for (int mt = 0; mt < kMaxTiles; ++mt) {
            if (mt < tiles) {
                load_words<WPT>(wb + (uint32_t)((16 * mt + g) * 128), g, h, t, xa[mt]);
                load_words<WPT>(wb + (uint32_t)((16 * mt + g + 8) * 128), g, h, t, xb[mt]);
            }
        }
#pragma unroll
        for (int i = 0; i < WPT; ++i) {
            uint32_t bo[NT][4];
#pragma unroll
            for (int u = 0; u < NT; ++u) {
                const uint4 r = av[u][i];
                bo[u][0] = __byte_perm(r.x, r.z, 0x5410);   // (a0, a4)
                bo[u][1] = __byte_perm(r.x, r.z, 0x7632);   // (a1, a5)
                bo[u][2] = __byte_perm(r.y, r.w, 0x5410);   // (a2, a6)
                bo[u][3] = __byte_perm(r.y, r.w, 0x7632);   // (a3, a7)
                mma_acc(sg[u][0], ONES, ONES, ONES, ONES, bo[u][0], bo[u][1]);
                mma_acc(sg[u][1], ONES, ONES, ONES, ONES, bo[u][2], bo[u][3]);
            }
#pragma unroll
            for (int mt = 0; mt < kMaxTiles; ++mt) {
                if (mt < tiles) {
                    const uint32_t a00 = pair128(xa[mt][i], 0), a01 = pair128(xb[mt][i], 0),
                                   a02 = pair128(xa[mt][i], 1), a03 = pair128(xb[mt][i], 1);
                    const uint32_t a10 = pair128(xa[mt][i], 2), a11 = pair128(xb[mt][i], 2),
                                   a12 = pair128(xa[mt][i], 3), a13 = pair128(xb[mt][i], 3);
#pragma unroll
                    for (int u = 0; u < NT; ++u) {
                        mma_acc(d[mt][u][0], a00, a01, a02, a03, bo[u][0], bo[u][1]);
                        mma_acc(d[mt][u][NCH - 1], a10, a11, a12, a13, bo[u][2], bo[u][3]);
                    }
                }
            }
        }
        // acc += s (D_g - (128 + z) S_g); -(128 + z) = (2^23 - 128) - (2^23 + z)
#pragma unroll
        for (int mt = 0; mt < kMaxTiles; ++mt) {
            if (mt < tiles) {
                float s[2], cz[2];
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int row = 16 * mt + g + 8 * half;
                    s[half] = __uint_as_float((uint32_t)sS[row * G + gi] << 16);
                    cz[half] = 8388480.f - __uint_as_float(0x4B000000u | (uint32_t)sZ[row * G + gi]);
                }
#pragma unroll
                for (int u = 0; u < NT; ++u)
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        acc[mt][u][e] = fmaf(s[e >> 1],
                                             fmaf(cz[e >> 1], sg[u][0][e] + sg[u][1][e],
                                                  NCH == 1 ? d[mt][u][0][e] : d[mt][u][0][e] + d[mt][u][NCH - 1][e]),
                                             acc[mt][u][e]);
            }
        }
    };

    // the warp's groups in order: every third group (from `half`) of the
    // stages pair, pair + 4, ...; each group's activations are loaded while the
    // previous group is multiplied
    const int pair = warp & 3, half = warp >> 2;   // set, member
    uint4 cur[NT][WPT], nxt[NT][WPT];
    if (pair < nch && pair * geo.nkb * GU + half < G) load_act(pair * geo.nkb * GU + half, cur);
#pragma unroll 1
    for (int ch = pair; ok && ch < nch; ch += kPairs) {
        const int s = slot(ch);
        if (!wait_bar_warp(FULL(s), (uint32_t)((ch / geo.stages) & 1), abort_flag, d_error)) {
            ok = false;
            break;
        }
        const uint32_t st = sbase + (uint32_t)(s * geo.stage_bytes);
        const int g0 = ch * geo.nkb * GU, g1 = std::min(G, (ch + 1) * geo.nkb * GU);   // the stage's groups
        const int gn = ch + kPairs < nch && (ch + kPairs) * geo.nkb * GU + half < G
                           ? (ch + kPairs) * geo.nkb * GU + half : -1;                    // the next stage's first
#pragma unroll 1
        for (int gi = g0 + half; gi < g1; gi += kPer) {
            const int next = gi + kPer < g1 ? gi + kPer : gn;
            if (next >= 0) load_act(next, nxt);
            group(st + (uint32_t)((gi - g0) / GU) * wbox, (gi - g0) % GU, gi, cur);
#pragma unroll
            for (int u = 0; u < NT; ++u)
#pragma unroll
                for (int i = 0; i < WPT; ++i) cur[u][i] = nxt[u][i];
        }
        arrive_warp(EMPTY(s));
    }

    // the twelve warps' sums of each output meet in shared memory
    constexpr int RC = 8 * NT;
    if (ok) {
        float *mine = red + warp * (16 * kMaxTiles * RC);
#pragma unroll
        for (int mt = 0; mt < kMaxTiles; ++mt) {
            if (mt < tiles) {
#pragma unroll
                for (int u = 0; u < NT; ++u) {
                    float *p = mine + (mt * 16 + g) * RC + u * 8 + 2 * t;
                    p[0] = acc[mt][u][0];
                    p[1] = acc[mt][u][1];
                    p[8 * RC] = acc[mt][u][2];
                    p[8 * RC + 1] = acc[mt][u][3];
                }
            }
        }
    }
    uint32_t rphase = 0;
    ok = group_sync_warp(REDB, rphase, abort_flag, d_error) && ok;
    if (!ok) return;
    constexpr int PER = 16 * kMaxTiles * RC;
    for (int idx = threadIdx.x; idx < rows * M; idx += kMmaWarps * 32) {
        const int m = idx / rows, r = idx - m * rows;
        const int o = r * RC + m;
        float v = red[o];
#pragma unroll
        for (int w = 1; w < kMmaWarps; ++w) v += red[w * PER + o];
        C[(int64_t)m * N + r0 + r] = f32_to_bf16_rn(v);
    }
}

// Geometry for M tokens on `grid` CTAs: false when a band would exceed
// kW4BandMaxRows rows, M exceeds kW4BandMaxTokens or K / group exceeds
// kW4BandMaxGroups.  A band that fits the budget whole goes in four stages
// (one per MMA warp, all requested at once); otherwise stages of as many
// 256-k boxes as eight slots fit.
bool w4band_geometry(int64_t M, int64_t N, int64_t K, int64_t group, int grid, W4BandGeo *g)
{
    if (M < 1 || M > kW4BandMaxTokens || N < 1 || K < 1 || grid < 1 || K % group) return false;
    const int64_t rows_max = (N + grid - 1) / grid;
    const int64_t G = K / group;
    if (rows_max > kW4BandMaxRows || G > kW4BandMaxGroups) return false;
    const int nt = w4band_nt(M);
    g->tiles = (int)((rows_max + 15) / 16);
    g->wrows = 16 * g->tiles;
    g->sz_bytes = (int)((g->wrows * G * 3 + 15) / 16 * 16);
    const int box = g->wrows * 128;
    const int kbs = (int)((K + kBoxK - 1) / kBoxK);
    const int budget = kSmemCap - g->sz_bytes - red_bytes(nt) - kBarBytes - 1024;
    if (kbs * box <= budget && kbs >= 4) {
        g->nkb = (kbs + 3) / 4;
        g->stages = (kbs + g->nkb - 1) / g->nkb;   // 4 (or fewer when the boxes divide unevenly)
    } else if (kbs < 4) {
        g->nkb = 1;
        g->stages = kbs;
    } else {
        g->nkb = std::max(1, std::min(kbs, budget / (kMaxStages * box)));
        const int nch = (kbs + g->nkb - 1) / g->nkb;
        g->stages = nch > 4 ? kMaxStages : nch;
    }
    g->stage_bytes = g->nkb * box;
    return g->stages * g->stage_bytes <= budget;
}

template <int NT, int WPT>
cudaError_t launch_t(const CUtensorMap &m, const CUtensorMap &m3, int three_d, const GemmArgs &a, const Plan &p,
                     const LaunchCtx &c, const W4BandGeo &g)
{
    auto kern = k_w4_band<NT, WPT>;
    static std::once_flag once[64];
    static cudaError_t attr_err[64];
    int dev = 0;
    cudaGetDevice(&dev);
    std::call_once(once[dev & 63], [&] {
        attr_err[dev & 63] = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemCap);
    });
    if (attr_err[dev & 63] != cudaSuccess) return attr_err[dev & 63];
    const int smem = w4band_smem(g, NT);
    if (smem > kSmemCap) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.grid, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = c.stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, m, m3, three_d, (const uint16_t *)a.A, (const uint16_t *)a.scales,
                              (const uint8_t *)a.zeros, (uint16_t *)a.C, (int)a.M, (int)a.N, (int)a.K, g, c.d_error,
                              g_debug_stall);
}

template <int NT>
cudaError_t launch_nt(const CUtensorMap &m, const CUtensorMap &m3, int three_d, const GemmArgs &a, const Plan &p,
                      const LaunchCtx &c, const W4BandGeo &g)
{
    switch (a.group) {
    case 32: return launch_t<NT, 1>(m, m3, three_d, a, p, c, g);
    case 64: return launch_t<NT, 2>(m, m3, three_d, a, p, c, g);
    default: return launch_t<NT, 4>(m, m3, three_d, a, p, c, g);
    }
}

}  // namespace

bool plan_w4_band(int64_t M, int64_t N, int64_t K, int64_t group, int sm_count, Plan *p)
{
    const int grid = (int)std::min<int64_t>(sm_count, N);
    W4BandGeo g;
    if (!w4band_geometry(M, N, K, group, grid, &g)) return false;
    p->variant = GEMM_VARIANT_BAND;
    p->kernels = 1;
    p->grid = grid;
    p->split = 1;
    p->tile_m = 8 * w4band_nt(M);
    p->tile_n = (int)((N + grid - 1) / grid);
    p->stages = g.stages;
    p->bn = kBoxK * g.nkb;   // k per stage
    p->mode = 0;
    return true;
}

cudaError_t launch_w4_band(const GemmArgs &a, const Plan &p, const LaunchCtx &c)
{
    W4BandGeo g;
    if (!w4band_geometry(a.M, a.N, a.K, a.group, p.grid, &g)) return cudaErrorInvalidValue;
    CUtensorMap m, m3;
    if (!make_map_words(&m, a.B, a.N, a.K, g.wrows)) return cudaErrorInvalidValue;
    const int three_d = a.K % kBoxK == 0 && make_map_words_kblocks(&m3, a.B, a.N, a.K, g.wrows, g.nkb);
    if (!three_d) m3 = m;
    return launch_nt<1>(m, m3, three_d, a, p, c, g);
}

}  // namespace dbw
