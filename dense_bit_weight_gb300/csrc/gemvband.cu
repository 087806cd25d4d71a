// gemvband.cu -- bf16 decode GEMM for up to 32 tokens: every SM streams one
// contiguous band of weight rows through a deep ring of TMA copies, and four
// warps multiply it with warp-level MMAs (mma.sync.m16n8k16, bf16 -> fp32;
// weight rows on the MMA's M side, tokens on its N side).
//
// The contraction is the decode GEMV of the hk-dsl PyPI page ("Results",
// kernels inside the engines: "decode GEMV, 1-32 tokens"): C[m, n] =
// sum_k A[m, k] B[n, k] with a handful of tokens, so the time is the weight
// stream.  What sets it at a few tens of MB per call is how soon every SM has
// its bytes in flight and how evenly the SMs finish:
//   - CTA c of G takes rows [c N / G, (c + 1) N / G) over all of K (a band of
//     at most 64 rows): the SMs' shares differ by one row, and no partial sum
//     ever leaves the SM (no workspace, no second pass, no cross-CTA wait);
//   - a stage is a k-chunk of the band: 64-k TMA boxes (128-byte swizzle)
//     of 16 * ceil(rows / 16) weight rows from the band's first row (the
//     rows past the band belong to the neighbouring band, which asks for
//     them at the same time, so they come from L2; their sums are dropped)
//     and of the tokens (rows past M, and k past K, read as zero), each
//     operand's boxes of a stage fetched by one 3-D copy when K is a multiple
//     of 64.  Few, large copies: with one bulk copy per row and k-chunk
//     (512-byte pieces) a call took ~40 ns per copy per SM, and with one 2-D
//     copy per 64-k box ~90 ns per copy, whatever its size;
//   - the ring holds about 190 KB per SM, all requested as soon as the grid
//     dependency is satisfied; before that wait the copy warp only asks L2
//     for the first stages;
//   - the four MMA warps take whole stages in turn (four stages multiplied at
//     once) and keep their own fp32 sums; the four sums of an output meet
//     once, in shared memory, added in warp order (deterministic), and leave
//     as bf16 with the bias epilogues applied in fp32.  (With the warps
//     sharing each stage's boxes instead, every stage cost a warp's whole
//     wait-load-multiply latency chain, ~0.55 us, whatever its size.)
// Every wait is bounded (waits.cuh); a copy warp that gives up drains the
// copies it issued before the CTA exits.
#include <cuda.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "waits.cuh"

namespace dbw {
namespace {

constexpr int kMmaWarps = 4;
constexpr int kThreads = (kMmaWarps + 1) * 32;   // + the copy warp
constexpr int kMaxTiles = kBandMaxRows / 16;      // 16-row MMA tiles per band
constexpr int kMaxStages = 8;
constexpr int kSmemCap = 200 * 1024;              // dynamic shared memory the kernel may take

struct BandGeo {
    int nkb;           // 64-k boxes per stage
    int stages;        // ring depth
    int wrows;         // weight rows per box: 16 * tiles
    int tiles;         // 16-row MMA tiles per box
    int stage_bytes;   // nkb * (wrows + 8 NT) * 128
};

constexpr int red_bytes(int nt) { return kMmaWarps * 16 * kMaxTiles * 8 * nt * 4; }

int band_nt(int64_t M) { return M <= 8 ? 1 : M <= 16 ? 2 : 4; }

int band_smem(const BandGeo &g, int nt)
{
    return g.stages * g.stage_bytes + red_bytes(nt) + 8 * (2 * kMaxStages + 2) + 1024;   // + alignment slack
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void mma_acc(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Shared-memory layout of a stage: the nkb weight boxes ([wrows][64] bf16,
// 128-byte rows, 16-byte piece c of row r at piece c ^ (r % 8)), then the nkb
// token boxes ([8 NT][64]).  Every box starts on a 1024-byte boundary.
template <int NT>
__global__ void __launch_bounds__(kThreads, 1)
k_gemv_band(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmA,
            const __grid_constant__ CUtensorMap tmW3, const __grid_constant__ CUtensorMap tmA3, int three_d,
            uint16_t *__restrict__ C, const uint16_t *__restrict__ bias, int epi, int M, int N, int K, int64_t ldc,
            BandGeo geo, int *__restrict__ d_error, int stall)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = ptx::smem_addr(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t *smem = smem_raw + (sbase - raw);
    const int ring = geo.stages * geo.stage_bytes;
    float *red = reinterpret_cast<float *>(smem + ring);
    const uint32_t bars = sbase + (uint32_t)(ring + red_bytes(NT));
    auto FULL = [&](int s) { return bars + 8u * (uint32_t)s; };
    auto EMPTY = [&](int s) { return bars + 8u * (uint32_t)(kMaxStages + s); };
    const uint32_t REDB = bars + 8u * (2 * kMaxStages);
    volatile uint32_t *abort_flag =
        reinterpret_cast<volatile uint32_t *>(smem + ring + red_bytes(NT) + 8 * (2 * kMaxStages + 1));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r0 = (int)((int64_t)blockIdx.x * N / gridDim.x);
    const int rows = (int)((int64_t)(blockIdx.x + 1) * N / gridDim.x - r0);
    const int kbs = (K + 63) / 64;                       // 64-k boxes over K
    const int nch = (kbs + geo.nkb - 1) / geo.nkb;       // stages over K
    const uint32_t wbox = (uint32_t)geo.wrows * 128u, abox = (uint32_t)NT * 1024u;
    const uint32_t act_off = (uint32_t)geo.nkb * wbox;   // token boxes after the weight boxes
    // Ring slot of stage ch.  MMA warp w consumes the stages ch = w mod 4, so
    // with 8 slots each warp owns slots w and w + 4 (with 4, slot w; with
    // fewer, every stage has its own slot): the previous use of a slot is
    // always the same warp's previous stage, and a parity wait can never see
    // a phase two steps away.  The use count of a slot is ch / stages.
    auto slot = [&](int ch) { return geo.stages >= 4 ? (ch & 3) + 4 * ((ch >> 2) % (geo.stages >> 2)) : ch; };

    if (threadIdx.x == 0) {
        for (int s = 0; s < geo.stages; ++s) {
            ptx::mbar_init(FULL(s), 1);
            ptx::mbar_init(EMPTY(s), 1);   // one MMA warp consumes a stage
        }
        ptx::mbar_init(REDB, kMmaWarps);
        *abort_flag = 0u;
        ptx::fence_mbar_init();
    }
    __syncthreads();

    if (warp == kMmaWarps) {
        // ---------------------------------------------------------------- copy warp
        if (lane == 0) {
            ptx::prefetch_tmap(three_d ? &tmW3 : &tmW);
            ptx::prefetch_tmap(three_d ? &tmA3 : &tmA);
            // before the dependency wait: ask L2 for the first stages' weights
            if (three_d) {
                for (int ch = 0; ch < std::min(nch, geo.stages); ++ch) ptx::tma_prefetch_l2_3d(&tmW3, 0, r0, ch * geo.nkb);
            } else {
                const int pre = std::min(kbs, geo.stages * geo.nkb);
                for (int b = 0; b < pre; ++b) ptx::tma_prefetch_l2_2d(&tmW, 64 * b, r0);
            }
        }
        ptx::pdl_wait();
        ptx::pdl_launch_dependents();
        const uint64_t pol_w = ptx::policy_evict_first(), pol_a = ptx::policy_evict_last();
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
                        // one copy per operand: all nkb boxes (past K: zeros)
                        ptx::mbar_arrive_expect_tx(FULL(s), (uint32_t)geo.nkb * (wbox + abox));
                        ptx::tma_load_3d(st, &tmW3, FULL(s), 0, r0, b0, pol_w);
                        ptx::tma_load_3d(st + act_off, &tmA3, FULL(s), 0, 0, b0, pol_a);
                    } else {
                        ptx::mbar_arrive_expect_tx(FULL(s), (uint32_t)nb * (wbox + abox));
                        for (int b = 0; b < nb; ++b) {
                            ptx::tma_load_2d(st + (uint32_t)b * wbox, &tmW, FULL(s), 64 * (b0 + b), r0, pol_w);
                            ptx::tma_load_2d(st + act_off + (uint32_t)b * abox, &tmA, FULL(s), 64 * (b0 + b), 0, pol_a);
                        }
                    }
                }
                __syncwarp();
                ++issued;
            }
        }
        // copies still in flight land before the CTA may exit (the last
        // `stages` issued chunks are the latest phase of their slots)
        if (lane == 0)
            for (int ch = std::max(0, issued - geo.stages); ch < issued; ++ch)
                wait_bar_drain(FULL(slot(ch)), (uint32_t)((ch / geo.stages) & 1));
        return;
    }

    // -------------------------------------------------------------------- MMA warps
    // warp w takes the stages w, w + 4, ... whole (the warps work on four
    // stages at once, so no warp's latency chain paces the stream); within a
    // stage its 64-k boxes alternate between two accumulator sets (NT <= 2)
    ptx::pdl_wait();
    const int tiles = (rows + 15) >> 4;   // this band's MMA tiles (<= geo.tiles)
    constexpr int SETS = NT <= 2 ? 2 : 1;
    float acc[SETS][kMaxTiles][NT][4];
#pragma unroll
    for (int q = 0; q < SETS; ++q)
#pragma unroll
        for (int i = 0; i < kMaxTiles; ++i)
#pragma unroll
            for (int j = 0; j < NT; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[q][i][j][e] = 0.f;
    // ldmatrix rows: A, x4 = rows 0-7 / 8-15 by lane octet, k pieces 2s / 2s + 1
    // by lane half; B (tokens), x4 = k pieces 2s .. 2s + 3 (two k-steps) by
    // lane octet.  A row's swizzle term is its index mod 8 = lane mod 8.
    const int sw = lane & 7;
    const uint32_t a_row = (uint32_t)(((lane & 7) + 8 * ((lane >> 3) & 1)) * 128);
    const int a_piece = lane >> 4;
    const uint32_t b_row = (uint32_t)((lane & 7) * 128);
    const int b_piece = lane >> 3;
    // one 64-k box into accumulator set q
    auto box = [&](uint32_t wb, uint32_t ab, float (&d)[kMaxTiles][NT][4]) {
#pragma unroll
        for (int s2 = 0; s2 < 2; ++s2) {   // pairs of k-steps: pieces 4 s2 .. 4 s2 + 3
            uint32_t bq[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
                ldsm_x4(ab + (uint32_t)(nt * 1024) + b_row + (uint32_t)(((4 * s2 + b_piece) ^ sw) << 4), bq[nt][0],
                        bq[nt][1], bq[nt][2], bq[nt][3]);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int piece = 4 * s2 + 2 * h + a_piece;
#pragma unroll
                for (int mt = 0; mt < kMaxTiles; ++mt) {
                    if (mt < tiles) {
                        uint32_t a0, a1, a2, a3;
                        ldsm_x4(wb + (uint32_t)(mt * 16 * 128) + a_row + (uint32_t)((piece ^ sw) << 4), a0, a1, a2,
                                a3);
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
                            mma_acc(d[mt][nt], a0, a1, a2, a3, bq[nt][2 * h], bq[nt][2 * h + 1]);
                    }
                }
            }
        }
    };
    bool ok = true;
#pragma unroll 1
    for (int ch = warp; ch < nch; ch += kMmaWarps) {
        const int s = slot(ch);
        if (!wait_bar_warp(FULL(s), (uint32_t)((ch / geo.stages) & 1), abort_flag, d_error)) {
            ok = false;
            break;
        }
        const int nb = std::min(geo.nkb, kbs - ch * geo.nkb);
        const uint32_t st = sbase + (uint32_t)(s * geo.stage_bytes);
#pragma unroll 1
        for (int b = 0; b < nb; b += SETS) {
            box(st + (uint32_t)b * wbox, st + act_off + (uint32_t)b * abox, acc[0]);
            if (SETS == 2 && b + 1 < nb)
                box(st + (uint32_t)(b + 1) * wbox, st + act_off + (uint32_t)(b + 1) * abox, acc[SETS - 1]);
        }
        arrive_warp(EMPTY(s));
    }
    if (SETS == 2) {
#pragma unroll
        for (int i = 0; i < kMaxTiles; ++i)
#pragma unroll
            for (int j = 0; j < NT; ++j)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[0][i][j][e] += acc[SETS - 1][i][j][e];
    }

    // the four warps' sums of each output meet in shared memory
    constexpr int RC = 8 * NT;   // token columns of the exchange
    const int g = lane >> 2, t = lane & 3;
    if (ok) {
        float *mine = red + warp * (16 * kMaxTiles * RC);
#pragma unroll
        for (int mt = 0; mt < kMaxTiles; ++mt) {
            if (mt < tiles) {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    float *p = mine + (mt * 16 + g) * RC + nt * 8 + 2 * t;
                    p[0] = acc[0][mt][nt][0];
                    p[1] = acc[0][mt][nt][1];
                    p[8 * RC] = acc[0][mt][nt][2];
                    p[8 * RC + 1] = acc[0][mt][nt][3];
                }
            }
        }
    }
    uint32_t rphase = 0;
    ok = group_sync_warp(REDB, rphase, abort_flag, d_error) && ok;
    if (!ok) return;
    constexpr int PER = 16 * kMaxTiles * RC;
    const bool has_bias = epi_has_bias(epi);
    for (int idx = threadIdx.x; idx < rows * M; idx += kMmaWarps * 32) {
        const int m = idx / rows, r = idx - m * rows;
        const int o = r * RC + m;
        float v = red[o];
#pragma unroll
        for (int w = 1; w < kMmaWarps; ++w) v += red[w * PER + o];
        if (has_bias) v = bias_act(v, bf16lo(bias[r0 + r]), epi);
        C[(int64_t)m * ldc + r0 + r] = f32_to_bf16_rn(v);
    }
}

}  // namespace

// Geometry of the band kernel for M tokens on `grid` CTAs: false when a band
// would exceed kBandMaxRows rows or M exceeds kBandMaxTokens.  The ring has
// eight stages (two per MMA warp; one per stage when K has at most four), a
// stage as many 64-k boxes as eight stages fit in the shared-memory budget.
static bool band_geometry(int64_t M, int64_t N, int64_t K, int grid, BandGeo *g)
{
    if (M < 1 || M > kBandMaxTokens || N < 1 || K < 1 || grid < 1) return false;
    const int64_t rows_max = (N + grid - 1) / grid;
    if (rows_max > kBandMaxRows) return false;
    const int nt = band_nt(M);
    g->tiles = (int)((rows_max + 15) / 16);
    g->wrows = 16 * g->tiles;
    const int box = (g->wrows + 8 * nt) * 128;   // one 64-k box of weights and tokens
    const int kbs = (int)((K + 63) / 64);
    const int budget = kSmemCap - red_bytes(nt) - 8 * (2 * kMaxStages + 2) - 1024;
    g->nkb = std::max(1, std::min(kbs, budget / (kMaxStages * box)));   // eight stages fit (a box is <= 12 KB)
    g->stage_bytes = g->nkb * box;
    const int nch = (kbs + g->nkb - 1) / g->nkb;
    g->stages = nch > 4 ? kMaxStages : nch;   // 8 (two slots per MMA warp), or one slot per stage
    return g->stages * g->stage_bytes <= budget;
}

bool plan_band(int64_t M, int64_t N, int64_t K, int sm_count, Plan *p)
{
    const int grid = (int)std::min<int64_t>(sm_count, N);
    BandGeo g;
    if (!band_geometry(M, N, K, grid, &g)) return false;
    p->variant = GEMM_VARIANT_BAND;
    p->kernels = 1;
    p->grid = grid;
    p->split = 1;
    p->tile_m = 8 * band_nt(M);
    p->tile_n = (int)((N + grid - 1) / grid);
    p->stages = g.stages;
    p->bn = 64 * g.nkb;   // k per stage
    p->mode = 0;
    return true;
}

cudaError_t launch_gemv_band(const GemmArgs &a, const Plan &p, const LaunchCtx &c)
{
    if (a.epi == GEMM_EPI_SILU_MUL || a.gends) return cudaErrorInvalidValue;
    if (epi_has_bias(a.epi) && !a.bias) return cudaErrorInvalidValue;
    BandGeo g;
    if (!band_geometry(a.M, a.N, a.K, p.grid, &g)) return cudaErrorInvalidValue;
    const int nt = band_nt(a.M);
    // K a multiple of 64: one 3-D copy per operand and stage; otherwise one
    // 2-D copy per 64-k box (the last box reads zeros past K)
    CUtensorMap mw, ma, mw3, ma3;
    if (!make_map_bf16(&mw, a.B, a.N, a.K, a.ldb, g.wrows) || !make_map_bf16(&ma, a.A, a.M, a.K, a.lda, 8 * nt))
        return cudaErrorInvalidValue;
    const int three_d = a.K % 64 == 0 && make_map_kblocks(&mw3, a.B, a.N, a.K, a.ldb, g.wrows, g.nkb) &&
                        make_map_kblocks(&ma3, a.A, a.M, a.K, a.lda, 8 * nt, g.nkb);
    if (!three_d) {
        mw3 = mw;
        ma3 = ma;
    }
    auto kern = nt == 1 ? k_gemv_band<1> : nt == 2 ? k_gemv_band<2> : k_gemv_band<4>;
    const int ki = nt == 1 ? 0 : nt == 2 ? 1 : 2;
    static std::once_flag once[3][64];
    static cudaError_t attr_err[3][64];
    int dev = 0;
    cudaGetDevice(&dev);
    std::call_once(once[ki][dev & 63], [&] {
        attr_err[ki][dev & 63] = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemCap);
    });
    if (attr_err[ki][dev & 63] != cudaSuccess) return attr_err[ki][dev & 63];
    const int smem = band_smem(g, nt);
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
    return cudaLaunchKernelEx(&cfg, kern, mw, ma, mw3, ma3, three_d, (uint16_t *)a.C, (const uint16_t *)a.bias, a.epi, (int)a.M,
                              (int)a.N, (int)a.K, a.ldc, g, c.d_error, g_debug_stall);
}

}  // namespace dbw
