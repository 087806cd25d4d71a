// umma.cu -- tcgen05 tensor-core GEMM for sm_103a.
//
// One persistent, warp-specialised kernel computes D = X . Y^T tile by tile,
// X and Y both K-contiguous bf16 ([rows, K] row-major), D accumulated in fp32
// in tensor memory (TMEM) and written as bf16:
//   prefill (X = A, Y = B):  D[i, j] = C[m0 + i, n0 + j]
//   skinny  (X = B, Y = A):  D[i, j] = C[m0 + j, n0 + i]   (swap AB: the weight
//            rows fill the 128-row side of the MMA, the few tokens its N side)
// The contraction is C[M,N] = A[M,K] . B[N,K]^T of the FlyDSL prebuilt
// kernels guide §3.1 (preshuffle GEMM); the design is the NVIDIA answer the
// HipKittens notes give for why producer/consumer specialisation pays on
// Blackwell (§2, the five reasons: TMA, tcgen05 reading shared/tensor memory,
// large shared memory, register reallocation, mbarriers).
//
// Warp roles (192 threads, one CTA per SM):
//   warp 0      TMA producer: loads a 128 x 64 X tile and a BN x 64 Y tile per
//               stage into a ring of shared-memory stages (128-byte swizzle),
//               signalling `full[s]` with the byte count
//   warp 1      allocates TMEM; one lane issues tcgen05.mma (M=128, N=BN,
//               K=16, four per stage) into one of two accumulators and
//               commits `empty[s]` (stage reusable) and `tfull[a]`
//   warps 2-5   epilogue: TMEM -> registers (tcgen05.ld 32x32b), bf16
//               round-to-nearest-even, global stores; release `tempty[a]`
// The two accumulators let the epilogue of one tile overlap the MMAs of the
// next (the prefetch-t+1-while-computing-t loop of the FlyDSL kernel
// authoring skill's "runtime loops" section, done by hardware queues here).
//
// Scheduling (the pages' split-K over CTAs only when the grid would underfill
// the device, FlyDSL prebuilt kernels guide §3c):
//   mode 0  whole tiles, CTA c takes tiles c, c+G, c+2G, ... in a grouped
//           raster (tile-rows in groups, so concurrently running CTAs share
//           operand tiles in L2 -- the L2-reuse window of the HipKittens
//           notes' Algorithm 1)
//   mode 1  stream-K: the (tile, k-block) units are cut into G contiguous
//           equal ranges, one per CTA.  A tile split across CTAs is summed by
//           whichever contributor arrives last: every contributor stores its
//           fp32 partial in the workspace, bumps the tile's counter, and the
//           last one adds all partials in increasing-k order (deterministic,
//           no float atomics) and resets the counter to zero.  Prefill
//           stream-K orders the tiles token-tile-row by row (raster groups of
//           one row) on a grid that is a multiple of the tile-rows: CTA c and
//           CTA c + G / rows then cover the same (weight tile, k-block) units
//           of neighbouring token tiles at the same time, and each weight
//           stage is read from HBM once.
//   mode 2  cluster split-K (decode): the S CTAs that split one tile's K
//           form a thread-block cluster, and CTA o owns row block o of the
//           tile.  Each CTA reads its fp32 partial from TMEM and sends every
//           row to the row's owner with 16-byte st.async remote stores into
//           slice `rank` of the owner's exchange region (bytes counted on the
//           owner's mbarrier); the owner sums its S slices in rank order
//           (deterministic, no global scratch), rounds to bf16 into a staging
//           tile and writes its block of C with one TMA store.  One tile per
//           CTA; the grid is small enough for every CTA to be resident at once.
//
// Launches use programmatic dependent launch: a kernel's prologue (barrier
// set-up, TMEM allocation, descriptor prefetch) overlaps the tail of the
// kernel before it, and it waits for that kernel before touching memory.
//
// Every mbarrier wait is bounded (1 s of %globaltimer).  On expiry the
// waiting thread raises a shared abort flag and the device error word; all
// roles leave their loops, the producer waits (bounded) for the copies it
// issued, the MMA lane for its issued MMAs, and TMEM is freed before exit.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "sched.cuh"
#include "waits.cuh"

namespace dbw {
namespace {

constexpr int BM = 128;          // MMA M: rows of X per tile
constexpr int BK = 64;           // k per MMA tile (one 128-byte swizzle row of bf16)
constexpr int kEpiThreads = 128;
constexpr int kDqThreads = 512;  // W4A16: dequantising threads (warps 6-21)
constexpr int kNX = 2;           // W4A16: dequantised 128 x 256 bf16 stages in TMEM (128 columns each)
constexpr uint32_t kXCol = 256;  // W4A16: TMEM column of the first dequantised stage
constexpr int kActWarp = 22;     // W4A16: warp that loads the activation tiles
__host__ __device__ constexpr int threads_for(bool w4) { return w4 ? 192 + kDqThreads + 32 : 192; }

// W4A16 operands beyond the packed-weight tensor map.
struct W4Args {
    const uint16_t *scales;      // bf16 [N, K/group]
    const uint8_t *zeros;        // uint8 [N, K/group]
    int K, G, group;
    int lg_group;                // log2(group); group is 32, 64 or 128
};

// store_chunk with a fused epilogue (a bias epilogue or GEMM_EPI_SILU_MUL).
// Rows of X (SWAP) or columns of Y hold weight rows; with GEMM_EPI_SILU_MUL
// they come as (gate, up) pairs 2j, 2j + 1 for output column j.  SWAP: a
// thread owns one weight row and its pair partner is the neighbouring lane
// (every lane of the warp must call this).  Kept out of line so the plain
// store path keeps its own register allocation.
template <bool SWAP>
__device__ __noinline__ void store_chunk_fused(uint16_t *__restrict__ C, int64_t ldc, int R, int Q, int r, int q0,
                                               const float *fin, const Sched &s)
{
    float f[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) f[j] = fin[j];
    if (s.epi == GEMM_EPI_SILU_MUL) {
        if (SWAP) {
            float u[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) u[j] = __shfl_down_sync(0xffffffffu, f[j], 1);
            if ((r & 1) == 0 && r < R) {
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    if (q0 + j < Q) C[(int64_t)(q0 + j) * ldc + (r >> 1)] = f32_to_bf16_rn(silu_mul(f[j], u[j]));
            }
        } else if (r < R) {
            float o[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) o[j] = silu_mul(f[2 * j], f[2 * j + 1]);
            uint16_t *dst = C + (int64_t)r * ldc + (q0 >> 1);
            if (q0 + 16 <= Q) {
                uint4 w;
                w.x = pack_bf16x2_rn(o[0], o[1]);
                w.y = pack_bf16x2_rn(o[2], o[3]);
                w.z = pack_bf16x2_rn(o[4], o[5]);
                w.w = pack_bf16x2_rn(o[6], o[7]);
                *reinterpret_cast<uint4 *>(dst) = w;
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (q0 + 2 * j < Q) dst[j] = f32_to_bf16_rn(o[j]);
            }
        }
        return;
    }
    if (epi_has_bias(s.epi)) {
        if (SWAP) {
            const float b = r < R ? bf16lo(s.bias[r]) : 0.f;
#pragma unroll
            for (int j = 0; j < 16; ++j) f[j] = bias_act(f[j], b, s.epi);
        } else {
#pragma unroll
            for (int j = 0; j < 16; ++j)
                if (q0 + j < Q) f[j] = bias_act(f[j], bf16lo(s.bias[q0 + j]), s.epi);
        }
    }
    store_chunk<SWAP>(C, ldc, R, Q, r, q0, f);
}

template <bool SWAP, bool FUSED>
__device__ __forceinline__ void store_chunk_epi(uint16_t *__restrict__ C, int64_t ldc, int R, int Q, int r, int q0,
                                                const float (&f)[16], const Sched &s)
{
    if (!FUSED || s.epi == GEMM_EPI_NONE) store_chunk<SWAP>(C, ldc, R, Q, r, q0, f);
    else store_chunk_fused<SWAP>(C, ldc, R, Q, r, q0, f, s);
}

// The cluster split-K reduction's store of one summed float4 (tokens q0 .. q0 + 3
// of row r) with a fused epilogue; paired: lanes rl, rl ^ 1 hold rows re, re + 1
// (every lane of the warp calls this).
template <bool SWAP>
__device__ __noinline__ void cluster_store_fused(uint16_t *__restrict__ C, int64_t ldc, int R, int Q, int r, int q0,
                                                 bool paired, bool odd, const float *ain, const Sched &s)
{
    float a[4] = {ain[0], ain[1], ain[2], ain[3]};
    if (paired) {
        float x[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) x[j] = __shfl_xor_sync(0xffffffffu, a[j], 1);
        const int re = r - (odd ? 1 : 0);   // the pair's even row
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {    // even lane: tokens 0, 1; odd lane: tokens 2, 3
            const int j = odd ? 2 + jj : jj;
            float lo = odd ? x[j] : a[j], hi = odd ? a[j] : x[j];
            const int q = q0 + j;
            if (q < Q && re < R) {
                if (s.epi == GEMM_EPI_SILU_MUL) {   // rows re, re + 1: gate and up of column re / 2
                    C[(int64_t)q * ldc + (re >> 1)] = f32_to_bf16_rn(silu_mul(lo, hi));
                    continue;
                }
                lo = bias_act(lo, bf16lo(s.bias[re]), s.epi);
                if (re + 1 < R) hi = bias_act(hi, bf16lo(s.bias[re + 1]), s.epi);
                uint16_t *dst = C + (int64_t)q * ldc + re;
                if (re + 1 < R) *reinterpret_cast<uint32_t *>(dst) = pack_bf16x2_rn(lo, hi);
                else *dst = f32_to_bf16_rn(lo);
            }
        }
    } else if (r < R && epi_has_bias(s.epi)) {   // (pairs are only split in twos)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int q = q0 + j;
            if (q < Q) {
                const float v = bias_act(a[j], bf16lo(s.bias[SWAP ? r : q]), s.epi);
                if (SWAP) C[(int64_t)q * ldc + r] = f32_to_bf16_rn(v);
                else C[(int64_t)r * ldc + q] = f32_to_bf16_rn(v);
            }
        }
    }
}

constexpr uint32_t tmem_cols_for(int n)
{
    return n <= 32 ? 32u : n <= 64 ? 64u : n <= 128 ? 128u : n <= 256 ? 256u : 512u;
}

// Shared memory.
// bf16: a ring of STAGES stages, each an X tile (128 x 64 bf16, 16 KB, TMA
// 128-B swizzle) and a Y tile (BN x 64 bf16).
// W4A16: two rings of 256-k stages.  Packed weights: STAGES stages of 128 rows
// of 4-bit codes (16 KB, TMA 128-B swizzle), released by the dequantising warps
// as soon as they have read them.  Activations: AST stages of four BN x 64 bf16
// tiles, released by the MMA.  The dequantised weights live in tensor memory
// (kNX stages of 128 x 256 bf16 from column kXCol), where the MMA reads its A
// operand.
// Cluster split-K (CS: the deep skinny instances): the S CTAs of a cluster
// exchange fp32 partial rows in a region of S slices of up to BM / S + 1 rows
// (slice s holds CTA s's rows for this CTA's block of the tile), followed by
// a bf16 staging tile for the TMA store of the block.  The region has its own
// shared memory when that fits beside the ring (RED_OWN: partials may arrive
// while this CTA is still in its main loop), otherwise it reuses the ring once
// every CTA of the cluster has drained its pipeline.
template <int BN, int STAGES, bool W4 = false, bool CS = false>
struct Layout {
    static constexpr int KSTAGE = W4 ? 4 * BK : BK;                 // k per ring stage
    static constexpr int X_BYTES = W4 ? BM * KSTAGE / 2 : BM * BK * 2;
    static constexpr int Y_BYTES = W4 ? 0 : BN * BK * 2;
    static constexpr int STAGE_BYTES = X_BYTES + Y_BYTES;
    static constexpr int AST = !W4 ? 0 : BN <= 16 ? 4 : BN <= 32 ? 3 : 2;
    static constexpr int A_BYTES = BN * KSTAGE * 2;                 // W4A16: one activation stage
    static constexpr int A_OFF = STAGES * STAGE_BYTES;
    static constexpr int SZ_OFF = A_OFF + AST * A_BYTES;   // end of the rings
    static constexpr int BAR_OFF = SZ_OFF;
    static constexpr int NBARS = 2 * STAGES + 6 + (W4 ? 2 * kNX + 2 * AST : 0);
    static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;
    // grouped GEMM (prefill kernel only): expert row ends [kMaxExperts], m-tile prefix [kMaxExperts + 1]
    static constexpr int GRP_OFF = MISC_OFF + 16;
    static constexpr int GRP_BYTES = (!W4 && BN == 256) ? (2 * kMaxExperts + 4) * 4 : 0;
    static constexpr int RSTRIDE = BN * 4 + 16;         // bytes per partial row (conflict-free 16-byte reads)
    static constexpr int RED_BYTES = CS ? (BM + 8) * RSTRIDE : 0;
    static constexpr int STG_BYTES = CS ? 64 * BN * 2 : 0;   // bf16 [BN][BM / S], S >= 2
    static constexpr int OWN_OFF = (GRP_OFF + GRP_BYTES + 127) / 128 * 128;
    static constexpr bool RED_OWN = CS && OWN_OFF + RED_BYTES + STG_BYTES + 1024 <= 227 * 1024;
    static constexpr int RED_OFF = RED_OWN ? OWN_OFF : 0;
    static constexpr int STG_OFF = RED_OFF + (RED_BYTES + 127) / 128 * 128;
    static constexpr int SMEM = (RED_OWN ? STG_OFF + STG_BYTES : GRP_OFF + GRP_BYTES) + 1024;   // + slack to align the base
    static_assert(!CS || RED_OWN || STG_OFF + STG_BYTES <= SZ_OFF, "the split-K region must fit the ring");
};

// FUSED: the instance serves gemm_bf16_fused (epilogues, gate/up pair maps);
// plain calls run the FUSED = false instances, which carry none of that code.
template <int BN, int STAGES, bool SWAP, int MINB, bool W4, bool FUSED>
__global__ void __launch_bounds__(threads_for(W4), MINB)
k_umma(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmY,
       const __grid_constant__ CUtensorMap tmC, uint16_t *__restrict__ C, int R, int Q, int64_t ldc, const Sched sched,
       float *__restrict__ ws, int *__restrict__ counters, int *__restrict__ d_error, const W4Args w4)
{
    using L = Layout<BN, STAGES, W4, SWAP && MINB == 1>;
    // W4A16 takes all 512 columns: two accumulators below kXCol, the
    // dequantised tiles above.  Its shared memory admits one CTA per SM, so
    // the allocation never waits on a CTA of the same cluster.
    constexpr uint32_t TMEM_COLS = W4 ? 512u : tmem_cols_for(2 * BN);
    static_assert(!W4 || (2 * BN <= (int)kXCol && kXCol + kNX * 128 <= 512), "W4A16 TMEM map");
    static_assert(!W4 || L::SMEM > 114 * 1024, "W4A16 needs one CTA per SM (it allocates all of TMEM)");
    constexpr uint32_t IDESC = ptx::idesc_bf16_f32(BM, BN);

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::BAR_OFF);
    uint32_t *misc = reinterpret_cast<uint32_t *>(smem + L::MISC_OFF);  // [0] tmem, [1] abort, [2] last flag
    const uint32_t sbase = ptx::smem_addr(smem);
    const uint32_t bar0 = ptx::smem_addr(bars);
    auto FULL = [&](int s) { return bar0 + 8u * s; };
    auto EMPTY = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto TFULL = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
    auto TEMPTY = [&](int a) { return bar0 + 8u * (2 * STAGES + 2 + a); };
    const uint32_t DONE = bar0 + 8u * (2 * STAGES + 4);
    const uint32_t REDUCE = bar0 + 8u * (2 * STAGES + 5);   // mode 2: incoming partial slices
    auto XFULL = [&](int b) { return bar0 + 8u * (2 * STAGES + 6 + b); };          // W4A16: dequantised tile ready
    auto XEMPTY = [&](int b) { return bar0 + 8u * (2 * STAGES + 6 + kNX + b); };   // W4A16: MMA done with it
    auto AFULL = [&](int a) { return bar0 + 8u * (2 * STAGES + 6 + 2 * kNX + a); };              // W4A16
    auto AEMPTY = [&](int a) { return bar0 + 8u * (2 * STAGES + 6 + 2 * kNX + L::AST + a); };   // W4A16

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    volatile uint32_t *abort_flag = misc + 1;
    // cluster split-K runs only in the deep skinny kernels (the planner never
    // asks another instance for it; they lack the shared memory for it)
    constexpr bool kCanClusterSplit = SWAP && MINB == 1;
    const bool cluster_split = kCanClusterSplit && sched.mode == 2 && sched.split > 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(FULL(s), 1);
            ptx::mbar_init(EMPTY(s), W4 ? kDqThreads / 32 : 1);   // W4A16: every dequantising warp releases
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(TFULL(a), 1);
            ptx::mbar_init(TEMPTY(a), kEpiThreads / 32);   // one arrival per epilogue warp
        }
        ptx::mbar_init(DONE, 1);
        ptx::mbar_init(REDUCE, 1);
        if (W4) {
            for (int b = 0; b < kNX; ++b) {
                ptx::mbar_init(XFULL(b), kDqThreads / 32);   // every dequantising warp
                ptx::mbar_init(XEMPTY(b), 1);
            }
            for (int a = 0; a < L::AST; ++a) {
                ptx::mbar_init(AFULL(a), 1);
                ptx::mbar_init(AEMPTY(a), 1);
            }
        }
        misc[1] = 0;
        misc[2] = 0;
        if (cluster_split) {   // this CTA's block receives S - 1 slices of BN fp32 per row
            const uint32_t rank = ptx::cluster_ctarank(), S = (uint32_t)sched.split;
            const uint32_t nrows = (rank + 1) * BM / S - rank * BM / S;
            ptx::mbar_arrive_expect_tx(REDUCE, (S - 1) * nrows * BN * 4);
        }
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_addr(misc), TMEM_COLS);
        ptx::tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tmX);
        ptx::prefetch_tmap(&tmY);
        if (sched.tma_c) ptx::prefetch_tmap(&tmC);
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = misc[0];
    // phase A of the cluster barrier: with its own region, a CTA may receive
    // partials as soon as every CTA's barriers are initialised
    if (L::RED_OWN && cluster_split) ptx::cluster_arrive();

    // Grouped GEMM (prefill kernel, whole tiles): expert g owns the token rows
    // [end[g-1], end[g]) of A and C and multiplies them by its weight rows
    // g*gN .. g*gN + gN - 1 of B.  The row ends come from the previous kernel
    // (a router), so every thread waits for it; warp 0 clamps them into a
    // non-decreasing sequence within [0, R] and writes the exclusive prefix of
    // the experts' m-tile counts; expert g then owns the tiles from
    // gpre[g] * tiles_q, m-tile fastest, and an expert with no rows owns none.
    int *gend = reinterpret_cast<int *>(smem + L::GRP_OFF);
    int *gpre = gend + kMaxExperts;
    int ntiles = sched.tiles;   // mode 0 tile count (the grouped GEMM finds its own here)
    if constexpr (L::GRP_BYTES > 0) {
        if (sched.gends) {
            ptx::pdl_wait();
            if (warp == 0) {
                const int G = sched.groups;
                const int per = (G + 31) / 32;   // consecutive experts per lane
                const int g0 = min(G, lane * per), g1 = min(G, g0 + per);
                int run = 0;                     // prefix max of the raw ends within this lane's run
                for (int g = g0; g < g1; ++g) run = max(run, __ldg(sched.gends + g));
                int before = run;                // inclusive max-scan over lanes, then shifted to exclusive
                for (int o = 1; o < 32; o <<= 1) {
                    const int v = __shfl_up_sync(0xffffffffu, before, o);
                    if (lane >= o) before = max(before, v);
                }
                before = __shfl_up_sync(0xffffffffu, before, 1);
                if (lane == 0) before = 0;
                int prev = min(before, R), mt = 0;
                run = before;
                for (int g = g0; g < g1; ++g) {
                    run = max(run, __ldg(sched.gends + g));
                    const int e = min(run, R);
                    gend[g] = e;
                    mt += (e - prev + BM - 1) / BM;
                    prev = e;
                }
                int base = mt;                   // exclusive sum-scan of the m-tile counts
                for (int o = 1; o < 32; o <<= 1) {
                    const int v = __shfl_up_sync(0xffffffffu, base, o);
                    if (lane >= o) base += v;
                }
                if (lane == 31) gpre[G] = base;
                base -= mt;
                prev = before < R ? before : R;
                for (int g = g0; g < g1; ++g) {
                    gpre[g] = base;
                    base += (gend[g] - (g == g0 ? prev : gend[g - 1]) + BM - 1) / BM;
                }
            }
            __syncthreads();
            ntiles = gpre[sched.groups] * sched.tiles_q;
        }
    }
    // tile t -> X rows from xrow, Y rows from yrow, C rows below rlim, C columns from qb
    auto geo = [&](int t, int &xrow, int &yrow, int &rlim, int &qb) {
        if (L::GRP_BYTES > 0 && sched.gends) {
            const int mt = t / sched.tiles_q;   // expert g owns tiles [gpre[g], gpre[g + 1]) * tiles_q
            int lo = 0, hi = sched.groups;   // the expert: largest lo < G with gpre[lo] <= mt
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (gpre[mid] <= mt) lo = mid;
                else hi = mid;
            }
            // within the expert, m-tiles vary fastest: the CTAs that read one
            // weight tile run side by side, so it comes from DRAM once
            const int nm = gpre[lo + 1] - gpre[lo];               // m-tiles of the expert
            const int local = t - gpre[lo] * sched.tiles_q;
            const int tqe = local / nm, mte = local - tqe * nm;
            xrow = (lo > 0 ? gend[lo - 1] : 0) + mte * BM;
            rlim = gend[lo];
            yrow = lo * sched.gN + tqe * BN;
            qb = tqe * BN;
        } else {
            int tr, tq;
            tile_coords(sched, t, tr, tq);
            xrow = tr * BM;
            yrow = tq * BN;
            rlim = R;
            qb = tq * BN;
        }
    };
    // Programmatic dependent launch: let the next kernel start its prologue now;
    // each role waits for the previous kernel (griddepcontrol.wait) just before
    // its first global-memory access.  The MMA role touches only shared and
    // tensor memory and does not wait.
    ptx::pdl_launch_dependents();

    bool have_acc = false;   // cluster split: this epilogue warp holds the tile's accumulator
    if (W4 && (warp == 0 || warp == kActWarp)) {
        // ------------------------------------------------------------ W4A16 producers
        // warp 0 streams the packed weights, warp kActWarp the activation tiles;
        // the two rings are independent so weight loads never wait on the MMA.
        if (lane == 0) {
            const bool packed = warp == 0;
            const uint64_t pol = packed ? ptx::policy_evict_first() : ptx::policy_evict_last();
            const int nslots = packed ? STAGES : L::AST;
            int slot = 0;
            uint32_t phase = 0;
            long long issued = 0;
            {
                SegIter pre(sched, blockIdx.x, ntiles);
                Segment s0;
                if (packed && pre.next(sched, s0) && !sched.stall) {
                    int tr, tq;
                    tile_coords(sched, s0.tile, tr, tq);
                    const int kend = min(s0.kb1, s0.kb0 + STAGES);
                    for (int kb = s0.kb0; kb < kend; ++kb) ptx::tma_prefetch_l2_2d(&tmX, kb * (L::KSTAGE / 8), tr * BM);
                }
                ptx::pdl_wait();
            }
            SegIter it(sched, blockIdx.x, ntiles);
            Segment seg;
            bool ok = true;
            while (ok && it.next(sched, seg)) {
                int tr, tq;
                tile_coords(sched, seg.tile, tr, tq);
                for (int kb = seg.kb0; kb < seg.kb1; ++kb) {
                    const uint32_t full = packed ? FULL(slot) : AFULL(slot);
                    const uint32_t empty = packed ? EMPTY(slot) : AEMPTY(slot);
                    if (!wait_bar(empty, phase ^ 1u, abort_flag, d_error)) {
                        ok = false;
                        break;
                    }
                    if (!sched.stall) {
                        if (packed) {
                            ptx::mbar_arrive_expect_tx(full, L::X_BYTES);
                            ptx::tma_load_2d(sbase + slot * L::STAGE_BYTES, &tmX, full, kb * (L::KSTAGE / 8),
                                             tr * BM, pol);
                        } else {   // four 64-k tiles, BN rows of 128 B each
                            ptx::mbar_arrive_expect_tx(full, L::A_BYTES);
                            for (int u = 0; u < L::KSTAGE / BK; ++u)
                                ptx::tma_load_2d(sbase + L::A_OFF + slot * L::A_BYTES + u * BN * BK * 2, &tmY, full,
                                                 kb * L::KSTAGE + u * BK, tq * BN, pol);
                        }
                        ++issued;
                    }
                    if (++slot == nslots) {
                        slot = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                for (int s = 0; s < nslots; ++s) {
                    if (issued <= s) continue;
                    const long long last = issued - 1 - ((issued - 1 - s) % nslots);
                    wait_bar_drain(packed ? FULL(s) : AFULL(s), (uint32_t)((last / nslots) & 1));
                }
            }
        }
    } else if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            // weights stream (evict first) unless several token tiles read them
            const bool y_once = !SWAP && sched.tiles_r == 1;
            const uint64_t pol_x = SWAP ? ptx::policy_evict_first() : ptx::policy_evict_last();
            const uint64_t pol_y = y_once ? ptx::policy_evict_first() : ptx::policy_evict_last();
            int stage = 0;
            uint32_t phase = 0;
            long long issued = 0;
            {
                // warm L2 with the first stages of this CTA's work while the
                // previous kernel drains, then wait for it
                SegIter pre(sched, blockIdx.x, ntiles);
                Segment s0;
                if (pre.next(sched, s0) && !sched.stall) {
                    int xrow, yrow, rlim, qb;
                    geo(s0.tile, xrow, yrow, rlim, qb);
                    const int kend = min(s0.kb1, s0.kb0 + STAGES);
                    for (int kb = s0.kb0; kb < kend; ++kb) {
                        if (FUSED && SWAP && sched.pairs) ptx::tma_prefetch_l2_3d(&tmX, kb * BK, 0, xrow / 2);
                        else ptx::tma_prefetch_l2_2d(&tmX, kb * BK, xrow);
                        if (FUSED && !SWAP && sched.pairs) ptx::tma_prefetch_l2_3d(&tmY, kb * BK, 0, yrow / 2);
                        else ptx::tma_prefetch_l2_2d(&tmY, kb * BK, yrow);
                    }
                }
                ptx::pdl_wait();
            }
            SegIter it(sched, blockIdx.x, ntiles);
            Segment seg;
            bool ok = true;
            while (ok && it.next(sched, seg)) {
                int xrow, yrow, rlim, qb;
                geo(seg.tile, xrow, yrow, rlim, qb);
                for (int kb = seg.kb0; kb < seg.kb1; ++kb) {
                    if (!wait_bar(EMPTY(stage), phase ^ 1u, abort_flag, d_error)) {
                        ok = false;
                        break;
                    }
                    if (!sched.stall) {
                        ptx::mbar_arrive_expect_tx(FULL(stage), (uint32_t)(sched.x_bytes + L::Y_BYTES));
                        const uint32_t xs = sbase + stage * L::STAGE_BYTES;
                        // (gate, up) pairs: the 3-D view [row / 2][gate or up][k] puts the
                        // pair's rows next to each other in the tile
                        if (FUSED && SWAP && sched.pairs) ptx::tma_load_3d(xs, &tmX, FULL(stage), kb * BK, 0, xrow / 2, pol_x);
                        else ptx::tma_load_2d(xs, &tmX, FULL(stage), kb * BK, xrow, pol_x);
                        if (FUSED && !SWAP && sched.pairs)
                            ptx::tma_load_3d(xs + L::X_BYTES, &tmY, FULL(stage), kb * BK, 0, yrow / 2, pol_y);
                        else ptx::tma_load_2d(xs + L::X_BYTES, &tmY, FULL(stage), kb * BK, yrow, pol_y);
                        ++issued;
                    }
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                // drain: every stage's most recent copy must land before exit
                for (int s = 0; s < STAGES; ++s) {
                    if (issued <= s) continue;
                    const long long last = issued - 1 - ((issued - 1 - s) % STAGES);
                    wait_bar_drain(FULL(s), (uint32_t)((last / STAGES) & 1));
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp runs the loop; one elected lane issues each MMA and
        // commit (see mma_bf16_warp).
        int stage = 0, acc = 0, xb = 0;
        uint32_t phase = 0, acc_phase = 0, xphase = 0;
        SegIter it(sched, blockIdx.x, ntiles);
        Segment seg;
        bool ok = true;
        while (ok && it.next(sched, seg)) {
            if (!wait_bar_warp(TEMPTY(acc), acc_phase ^ 1u, abort_flag, d_error)) break;
            ptx::tc_fence_after();
            const uint32_t d = tmem + (uint32_t)(acc * BN);
            if (W4) {
                // W4A16: per 256-k stage, one wait: the dequantising threads arrive on
                // XFULL only after their weights are in TMEM and the stage's
                // activations have landed (they wait for AFULL themselves), so the
                // 16 MMAs of a stage run back to back.  Each synchronisation point
                // of the issuing warp costs about as much as four N = 16 MMAs.
                // The next stage's XFULL is probed (non-blocking) before the last
                // sub-tile's MMAs and settled at the top of the next iteration, so
                // the barrier's latency overlaps MMA execution.
                bool probe = false;
                for (int kb = seg.kb0; kb < seg.kb1; ++kb) {
                    if (!settle_warp(probe, XFULL(xb), xphase, abort_flag, d_error)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t xa = tmem + kXCol + (uint32_t)(xb * 128);
                    const uint32_t ab = sbase + L::A_OFF + stage * L::A_BYTES;
                    const int nxb = xb + 1 == kNX ? 0 : xb + 1;
                    const uint32_t nxphase = nxb == 0 ? xphase ^ 1u : xphase;
#pragma unroll
                    for (int u = 0; u < L::KSTAGE / BK; ++u) {
                        if (u == L::KSTAGE / BK - 1)
                            probe = kb + 1 < seg.kb1 && ptx::mbar_test_wait(XFULL(nxb), nxphase);
                        const uint64_t bd = ptx::sdesc_kmajor_sw128(ab + u * BN * BK * 2);
#pragma unroll
                        for (int k = 0; k < BK / 16; ++k)   // 16 k = 8 TMEM columns of A, 32 bytes of B
                            ptx::mma_bf16_ts_warp(d, xa + (uint32_t)(32 * u + 8 * k), bd + 2u * k, IDESC,
                                                  (kb > seg.kb0 || u > 0 || k > 0) ? 1u : 0u);
                    }
                    ptx::mma_commit_warp(XEMPTY(xb));
                    ptx::mma_commit_warp(AEMPTY(stage));
                    if (++xb == kNX) {
                        xb = 0;
                        xphase ^= 1u;
                    }
                    if (++stage == L::AST) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            } else {
                for (int kb = seg.kb0; kb < seg.kb1; ++kb) {
                    if (!wait_bar_warp(FULL(stage), phase, abort_flag, d_error)) {
                        ok = false;
                        break;
                    }
                    const uint32_t xs = sbase + stage * L::STAGE_BYTES;
                    ptx::tc_fence_after();
                    const uint64_t ad = ptx::sdesc_kmajor_sw128(xs);
                    const uint64_t bd = ptx::sdesc_kmajor_sw128(xs + L::X_BYTES);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k)   // +32 bytes along K per step
                        ptx::mma_bf16_warp(d, ad + 2u * k, bd + 2u * k, IDESC, (kb > seg.kb0 || k > 0) ? 1u : 0u);
                    ptx::mma_commit_warp(EMPTY(stage));
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) break;
            ptx::mma_commit_warp(TFULL(acc));
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        ptx::mma_commit_warp(DONE);          // every issued MMA retires before TMEM is freed
        wait_bar_drain(DONE, 0);
    } else if (W4 && warp >= 6) {
        // ------------------------------------------------------------ W4A16 dequantisation
        // Warps 6-21: group u = (warp - 6) / 4 owns the 64-k sub-tile u of every
        // 256-k stage, and lane l of warp w the weight row 32 (w % 4) + l, which is
        // the TMEM lane that warp may write.  A thread reads its row's 8 packed
        // words (two 16-byte pieces of the 128-B-swizzled stage; every
        // quarter-warp touches eight consecutive rows, so the loads are free of
        // bank conflicts), releases the stage, computes w = (q - z) * s in bf16
        // and stores the row's 64 weights into sub-tile u of a TMEM stage buffer
        // as 32 columns of k pairs -- the A layout the MMA reads.  Within each
        // 8-k block the pairs are (k, k + 4), k = 0..3, as two nibbles one 16-bit
        // half apart extract with one shift and one mask; the activations are
        // copied into the same k order beforehand (k_permute_k8), so the MMA's
        // sum runs over the same products.  Before it
        // signals the MMA it also waits for the stage's activations, so the MMA
        // warp waits once per stage.
        //   128 + q is exact in bf16 as (0x4300 | q); subtracting 128 + z is
        //   exact (|q - z| <= 15); the product with s is rounded once (RNE).
        const int u = (warp - 6) >> 2;
        const int q4 = warp & 3;
        const int r = 32 * q4 + lane;
        const uint32_t pk_off0 = (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + (((2 * u) ^ (r & 7)) << 4));
        const uint32_t pk_off1 = (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + (((2 * u + 1) ^ (r & 7)) << 4));
        const uint32_t trow = tmem + ((uint32_t)(32 * q4) << 16) + kXCol;
        ptx::pdl_wait();                           // scales and zeros come from global memory
        int stage = 0, xsel = 0, astage = 0;
        uint32_t phase = 0, xphase = 0, aphase = 0;
        SegIter it(sched, blockIdx.x, ntiles);
        Segment seg;
        bool ok = true;
        while (ok && it.next(sched, seg)) {
            int tr, tq;
            tile_coords(sched, seg.tile, tr, tq);
            const int n = tr * BM + r;
            const bool nv = n < R;
            const uint16_t *srow = w4.scales + (int64_t)n * w4.G;
            const uint8_t *zrow = w4.zeros + (int64_t)n * w4.G;
            // (scale, zero) of the groups covering this thread's two 32-k halves
            // (different groups when g = 32), one stage ahead, through L1.  A half
            // at or beyond K gets scale 0 (its activations are zero-filled too).
            auto load_sz = [&](int kb, uint32_t &s0, uint32_t &z0, uint32_t &s1, uint32_t &z1) {
                const int k0 = kb * L::KSTAGE + u * BK;
                const bool in0 = nv && k0 < w4.K, in1 = nv && k0 + 32 < w4.K;
                const int g0 = k0 >> w4.lg_group, g1 = (k0 + 32) >> w4.lg_group;
                s0 = in0 ? __ldg(srow + g0) : 0u;
                z0 = in0 ? __ldg(zrow + g0) : 0u;
                if (g1 != g0 || !in1) {
                    s1 = in1 ? __ldg(srow + g1) : 0u;
                    z1 = in1 ? __ldg(zrow + g1) : 0u;
                } else {
                    s1 = s0;
                    z1 = z0;
                }
            };
            uint32_t s0, z0, s1, z1;
            load_sz(seg.kb0, s0, z0, s1, z1);
            // Barriers are probed (non-blocking) ahead of the arithmetic and settled
            // where their data is needed, so their latency overlaps the work.
            bool pfull = false;   // probe of this stage's FULL, taken in the previous iteration
            for (int kb = seg.kb0; kb < seg.kb1; ++kb) {
                uint32_t ns0 = 0, nz0 = 0, ns1 = 0, nz1 = 0;
                if (kb + 1 < seg.kb1) load_sz(kb + 1, ns0, nz0, ns1, nz1);
                if (!settle_warp(pfull, FULL(stage), phase, abort_flag, d_error)) {
                    ok = false;
                    break;
                }
                const uint32_t sb = sbase + stage * L::STAGE_BYTES;
                const uint4 wa = ptx::lds128(sb + pk_off0);
                const uint4 wb = ptx::lds128(sb + pk_off1);
                arrive_warp(EMPTY(stage));               // the packed stage may be refilled now
                const int nstage = stage + 1 == STAGES ? 0 : stage + 1;
                const uint32_t nphase = nstage == 0 ? phase ^ 1u : phase;
                const bool pxe = ptx::mbar_test_wait(XEMPTY(xsel), xphase ^ 1u);
                const bool pact = ptx::mbar_test_wait(AFULL(astage), aphase);
                pfull = kb + 1 < seg.kb1 && ptx::mbar_test_wait(FULL(nstage), nphase);
                const uint32_t words[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
                uint32_t v[2][16];
#pragma unroll
                for (int h = 0; h < 2; ++h) {          // 32 k = 16 columns per store
                    const uint32_t s2u = (h == 0 ? s0 : s1) * 0x00010001u;
                    const __nv_bfloat162 s2 = *reinterpret_cast<const __nv_bfloat162 *>(&s2u);
                    const uint32_t zbu = (0x4300u + (h == 0 ? z0 : z1)) * 0x00010001u;   // bf16x2 (128 + z)
                    const __nv_bfloat162 z2 = *reinterpret_cast<const __nv_bfloat162 *>(&zbu);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const uint32_t x = words[4 * h + j];
#pragma unroll
                        for (int jj = 0; jj < 4; ++jj) {   // column 4j + jj = (k jj, k jj+4) of this 8-k block
                            const uint32_t t = ((x >> (4 * jj)) & 0x000F000Fu) | 0x43004300u;   // bf16x2 128 + q
                            __nv_bfloat162 w2 = *reinterpret_cast<const __nv_bfloat162 *>(&t);
                            w2 = __hmul2(__hsub2(w2, z2), s2);
                            v[h][4 * j + jj] = *reinterpret_cast<const uint32_t *>(&w2);
                        }
                    }
                }
                if (!settle_warp(pxe, XEMPTY(xsel), xphase ^ 1u, abort_flag, d_error)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                ptx::tmem_st16(trow + (uint32_t)(xsel * 128 + u * 32), v[0]);
                ptx::tmem_st16(trow + (uint32_t)(xsel * 128 + u * 32 + 16), v[1]);
                ptx::tmem_wait_st();
                if (!settle_warp(pact, AFULL(astage), aphase, abort_flag, d_error)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_before();              // the MMA reads these columns after XFULL
                arrive_warp(XFULL(xsel));
                s0 = ns0;
                z0 = nz0;
                s1 = ns1;
                z1 = nz1;
                if (++xsel == kNX) {
                    xsel = 0;
                    xphase ^= 1u;
                }
                if (++astage == L::AST) {
                    astage = 0;
                    aphase ^= 1u;
                }
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
    } else if (warp >= 2 && warp < 6) {
        // ------------------------------------------------------------ epilogue
        const int q4 = warp & 3;            // TMEM lane quarter this warp may read
        const int row = q4 * 32 + lane;     // accumulator row
        const int etid = threadIdx.x - 64;  // 0..127
        ptx::pdl_wait();                    // C, workspace and counters may be in use by the previous kernel
        int acc = 0;
        uint32_t acc_phase = 0;
        SegIter it(sched, blockIdx.x, ntiles);
        Segment seg;
        while (it.next(sched, seg)) {
            if (!wait_bar_warp(TFULL(acc), acc_phase, abort_flag, d_error)) break;
            ptx::tc_fence_after();
            if (cluster_split) {   // one tile per CTA: its partial leaves from TMEM in the cluster tail
                have_acc = true;
                break;
            }
            int xrow, yrow, rlim, qb;
            geo(seg.tile, xrow, yrow, rlim, qb);
            const int r = xrow + row;
            const uint32_t taddr = tmem + ((uint32_t)(q4 * 32) << 16) + (uint32_t)(acc * BN);
            const bool whole = seg.kb0 == 0 && seg.kb1 == sched.nk;
            // stream-K partial: float4 columns, [column/4][row], so a warp's store is 512 contiguous bytes
            float4 *part = reinterpret_cast<float4 *>(ws) + (int64_t)(blockIdx.x * 2 + seg.slot) * (BM * BN / 4);
#pragma unroll 1
            for (int c = 0; c < BN; c += 16) {
                uint32_t v[16];
                __syncwarp();
                ptx::tmem_ld16(taddr + (uint32_t)c, v);
                ptx::tmem_wait_ld();
                float f[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) f[j] = __uint_as_float(v[j]);
                if (whole) {
                    store_chunk_epi<SWAP, FUSED>(C, ldc, rlim, Q, r, qb + c, f, sched);
                } else {
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        __stcg(part + (c / 4 + u) * BM + row,
                               make_float4(f[4 * u], f[4 * u + 1], f[4 * u + 2], f[4 * u + 3]));
                }
            }
            ptx::tc_fence_before();
            arrive_warp(TEMPTY(acc));
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
            if (whole) continue;

            // ---- stream-K fixup: the last contributor of this tile sums the partials
            const int t = seg.tile;
            const int c_first = cta_of_unit(sched, (long long)t * sched.nk);
            const int c_last = cta_of_unit(sched, (long long)(t + 1) * sched.nk - 1);
            __threadfence();
            ptx::named_bar_sync(1, kEpiThreads);
            if (etid == 0) {
                const int old = atomicAdd(counters + t, 1);
                const bool last = old == c_last - c_first;
                if (last) counters[t] = 0;
                misc[2] = last ? 1u : 0u;
            }
            ptx::named_bar_sync(1, kEpiThreads);
            if (!misc[2]) continue;
            __threadfence();
            constexpr int INFL = W4 ? 4 : (MINB == 1 ? 32 : 16);
            streamk_fixup<BN, INFL>(sched, ws, t, row, [&](int c0, const float(&f)[16]) {
                store_chunk_epi<SWAP, FUSED>(C, ldc, rlim, Q, r, qb + c0, f, sched);
            });
        }
    }

    if (cluster_split) {
        // Cluster split-K reduction.  CTA `rank` owns rows [r0, r1) of the tile:
        // every CTA sends those rows of its partial to the owner (slice `rank`
        // of the owner's region), the owner sums the S slices in rank order
        // (increasing k) and stores its block of C.
        const int S = sched.split;
        const int rank = (int)ptx::cluster_ctarank();
        const int nmax = (BM + S - 1) / S;                    // rows per owner, at most
        const int r0 = rank * BM / S, r1 = (rank + 1) * BM / S, nrows = r1 - r0;
        const bool epi = warp >= 2 && warp < 6;
        // phase A: every CTA's barriers are initialised (own region) or every
        // CTA's pipeline has drained, so the ring may take the partials
        if (!L::RED_OWN) ptx::cluster_arrive();
        ptx::cluster_wait();
        __syncwarp();   // (the cluster barrier's wait is per thread)
        const uint32_t red = sbase + (uint32_t)L::RED_OFF;
        if (epi && have_acc) {
            const int q4 = warp & 3;
            const int row = q4 * 32 + lane;                   // accumulator row (TMEM lane)
            const int o = ((row + 1) * S - 1) / BM;           // its owner: o * BM / S <= row < (o + 1) * BM / S
            const int o0 = o * BM / S;
            const uint32_t dst_local = red + (uint32_t)((rank * nmax + row - o0) * L::RSTRIDE);
            const uint32_t dst = o == rank ? dst_local : ptx::map_cluster(dst_local, (uint32_t)o);
            const uint32_t bar = ptx::map_cluster(REDUCE, (uint32_t)o);
            const uint32_t taddr = tmem + ((uint32_t)(q4 * 32) << 16);
            constexpr int CH = BN >= 32 ? 2 : 1;   // 16-column TMEM loads in flight together
#pragma unroll 1
            for (int c = 0; c < BN; c += 16 * CH) {
                uint32_t v[CH][16];
                __syncwarp();
#pragma unroll
                for (int h = 0; h < CH; ++h) ptx::tmem_ld16(taddr + (uint32_t)(c + 16 * h), v[h]);
                ptx::tmem_wait_ld();
#pragma unroll
                for (int h = 0; h < CH; ++h)
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const uint4 w = make_uint4(v[h][4 * u], v[h][4 * u + 1], v[h][4 * u + 2], v[h][4 * u + 3]);
                        const uint32_t off = (uint32_t)((c + 16 * h + 4 * u) * 4);
                        if (o == rank) ptx::sts128(dst + off, w);
                        else ptx::st_async_v4(dst + off, w, bar);
                    }
            }
            ptx::tc_fence_before();
        }
        bool ok = true;
        if (epi) {
            ok = wait_bar_warp(REDUCE, 0, abort_flag, d_error) && have_acc;   // warp-uniform: shuffles below
            ptx::named_bar_sync(1, kEpiThreads);                               // this CTA's own slice is written
        }
        // phase B: this CTA has received every byte sent to it, so no CTA leaves
        // while another still writes into its shared memory
        ptx::cluster_arrive();
        if (epi) {
            int tr, tq;
            tile_coords(sched, (int)blockIdx.x / S, tr, tq);
            const int qb = tq * BN;
            // thread -> (row rl, first float4 column c4); rows per owner padded to a
            // power of two so the mapping is shifts and masks
            const int etid = threadIdx.x - 64;
            const int lg = nrows <= 16 ? 4 : nrows <= 32 ? 5 : nrows <= 64 ? 6 : 7;
            const int rl = etid & ((1 << lg) - 1);   // neighbouring threads: neighbouring rows
            const int cstep = kEpiThreads >> lg;
            const uint32_t src = red + (uint32_t)(rl * L::RSTRIDE);
            const uint32_t stg = sbase + (uint32_t)L::STG_OFF;
            const bool tma = sched.tma_c != 0;
            // S in {2, 4, 8}: the owner's rows are a power of two and start even, every
            // lane of a warp runs the same iterations, and neighbouring lanes (rows r,
            // r + 1) pair their values into 4-byte stores of C
            const bool paired = SWAP && (S == 2 || S == 4 || S == 8);
            for (int c4 = etid >> lg; ok && rl < nrows && c4 < BN / 4; c4 += cstep) {
                uint4 u[8];
#pragma unroll
                for (int q = 0; q < 8; ++q)   // all slices' loads in flight before the sums
                    if (q < S) u[q] = ptx::lds128(src + (uint32_t)(q * nmax * L::RSTRIDE + c4 * 16));
                float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int q = 0; q < 8; ++q) {   // rank order
                    if (q < S) {
                        a[0] += __uint_as_float(u[q].x);
                        a[1] += __uint_as_float(u[q].y);
                        a[2] += __uint_as_float(u[q].z);
                        a[3] += __uint_as_float(u[q].w);
                    }
                }
                const int r = tr * BM + r0 + rl;
                if (tma) {   // bf16 [token][row] staging tile of the TMA store
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        ptx::sts16(stg + (uint32_t)(((c4 * 4 + j) * nrows + rl) * 2), f32_to_bf16_rn(a[j]));
                } else if (FUSED && sched.epi != GEMM_EPI_NONE) {
                    cluster_store_fused<SWAP>(C, ldc, R, Q, r, qb + c4 * 4, paired, rl & 1, a, sched);
                } else if (paired) {
                    float x[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) x[j] = __shfl_xor_sync(0xffffffffu, a[j], 1);
                    const bool odd = rl & 1;
                    const int re = r - (odd ? 1 : 0);   // the pair's even row
#pragma unroll
                    for (int jj = 0; jj < 2; ++jj) {    // even lane: tokens 0, 1; odd lane: tokens 2, 3
                        const int j = odd ? 2 + jj : jj;
                        const float lo = odd ? x[j] : a[j], hi = odd ? a[j] : x[j];
                        const int q = qb + c4 * 4 + j;
                        if (q < Q && re < R) {
                            uint16_t *dst = C + (int64_t)q * ldc + re;
                            if (re + 1 < R) *reinterpret_cast<uint32_t *>(dst) = pack_bf16x2_rn(lo, hi);
                            else *dst = f32_to_bf16_rn(lo);
                        }
                    }
                } else if (r < R) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int q = qb + c4 * 4 + j;
                        if (q < Q) {
                            if (SWAP) C[(int64_t)q * ldc + r] = f32_to_bf16_rn(a[j]);
                            else C[(int64_t)r * ldc + q] = f32_to_bf16_rn(a[j]);
                        }
                    }
                }
            }
            if (tma) {   // (every epilogue warp reaches the barrier, whatever its `ok`)
                ptx::fence_proxy_async_smem();   // the staging tile is read by the TMA engine
                __syncwarp();
                ptx::named_bar_sync(1, kEpiThreads);
                if (etid == 0 && ok) {            // box: nrows rows of C's columns x BN tokens (clipped)
                    ptx::tma_store_2d(&tmC, stg, tr * BM + r0, qb);
                    ptx::bulk_commit_group();
                    ptx::bulk_wait_group_read0();
                }
            }
        }
        ptx::cluster_wait();
    }

    // every warp converged before the CTA barrier (bar.sync counts warps; a
    // warp split by the per-thread cluster wait or an elected branch would
    // otherwise arrive in pieces)
    __syncwarp();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ------------------------------------------------------------------ host side

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// [rows, K] bf16 row-major with leading dimension ld (elements); box 64 x box_rows,
// 128-byte swizzle, out-of-range elements read as zero.
bool make_map(CUtensorMap *m, const void *ptr, int64_t rows, int64_t K, int64_t ld, int box_rows)
{
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
    cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}


// C of the skinny kernels ([Q tokens][R columns] bf16, row pitch ldc) for the
// cluster split-K's TMA store: a box of BM / S columns x bn tokens, no swizzle.
// Used when the box is a whole number of 16-byte units (S = 2, 4 or 8) and the
// result needs no epilogue; otherwise the kernel stores directly.
bool cluster_store_map(CUtensorMap *m, Sched &s, const Plan &p, void *C, int64_t R, int64_t Q, int64_t ldc)
{
    s.tma_c = 0;
    const int S = p.split;
    if (p.variant != GEMM_VARIANT_SKINNY || p.mode != 2 || p.ctas_per_sm != 1 || s.epi != GEMM_EPI_NONE) return false;
    if ((S != 2 && S != 4 && S != 8) || (reinterpret_cast<uintptr_t>(C) & 15) || (ldc * 2) % 16) return false;
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)R, (cuuint64_t)Q};
    cuuint64_t strides[1] = {(cuuint64_t)ldc * 2};
    cuuint32_t box[2] = {(cuuint32_t)(BM / S), (cuuint32_t)p.bn};
    cuuint32_t estr[2] = {1, 1};
    if (fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, C, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
           CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
        CUDA_SUCCESS)
        return false;
    s.tma_c = 1;
    return true;
}

// Packed 4-bit weights for the tcgen05 kernel: boxes of 32 words x 128 rows.
bool make_map_packed(CUtensorMap *m, const void *ptr, int64_t rows, int64_t K)
{
    return make_map_words(m, ptr, rows, K, BM);
}

template <int BN, int STAGES, bool SWAP, int MINB, bool W4 = false, bool FUSED = false>
cudaError_t launch_t(const CUtensorMap &mx, const CUtensorMap &my, const CUtensorMap &mc, uint16_t *C, int R, int Q,
                     int64_t ldc, const Sched &s, const LaunchCtx &c, const W4Args &w4 = W4Args{})
{
    using L = Layout<BN, STAGES, W4, SWAP && MINB == 1>;
    auto kern = k_umma<BN, STAGES, SWAP, MINB, W4, FUSED>;
    static std::once_flag once[64];
    static cudaError_t attr_err[64];
    int dev = 0;
    cudaGetDevice(&dev);
    std::call_once(once[dev & 63], [&] {
        attr_err[dev & 63] = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
    });
    if (attr_err[dev & 63] != cudaSuccess) return attr_err[dev & 63];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)s.grid, 1, 1);
    cfg.blockDim = dim3(threads_for(W4), 1, 1);
    cfg.dynamicSmemBytes = L::SMEM;
    cfg.stream = c.stream;
    cudaLaunchAttribute at[2];
    int na = 0;
    at[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    if (s.mode == 2 && s.split > 1) {
        at[na].id = cudaLaunchAttributeClusterDimension;
        at[na].val.clusterDim.x = (unsigned)s.split;
        at[na].val.clusterDim.y = 1;
        at[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = at;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kern, mx, my, mc, C, R, Q, ldc, s, c.workspace, c.counters, c.d_error, w4);
}

}  // namespace

// Fused gate/up weights [2N, K] bf16 (gate rows 0..N-1, up rows N..2N-1) as
// the 3-D view [N][2][K]: a box of 64 k x 2 x box_pairs puts the gate and up
// rows of output column j next to each other (rows 2j, 2j + 1 of the tile),
// 128-byte swizzle as make_map.
bool make_map_pairs(CUtensorMap *m, const void *ptr, int64_t N, int64_t K, int64_t ld, int box_pairs)
{
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)K, 2, (cuuint64_t)N};
    cuuint64_t strides[2] = {(cuuint64_t)(N * ld * 2), (cuuint64_t)ld * 2};
    cuuint32_t box[3] = {(cuuint32_t)BK, 2, (cuuint32_t)box_pairs};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// bf16 [rows, K] (K a multiple of 64, leading dimension ld) as the 3-D view
// [K / 64][rows][64]: one box of box_kb 64-k blocks x box_rows rows lands as
// box_kb consecutive [box_rows][64] tiles (128-byte swizzle), the layout of
// box_kb separate 2-D boxes of make_map_bf16, in one copy.
bool make_map_kblocks(CUtensorMap *m, const void *ptr, int64_t rows, int64_t K, int64_t ld, int box_rows, int box_kb)
{
    if (K % BK) return false;
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {(cuuint64_t)BK, (cuuint64_t)rows, (cuuint64_t)(K / BK)};
    cuuint64_t strides[2] = {(cuuint64_t)ld * 2, (cuuint64_t)BK * 2};
    cuuint32_t box[3] = {(cuuint32_t)BK, (cuuint32_t)box_rows, (cuuint32_t)box_kb};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// C [rows, cols] bf16 for TMA stores of 32 rows x 16 columns with the
// 32-byte swizzle; elements beyond the extents are not written.
bool make_map_c16(CUtensorMap *m, void *C, int64_t rows, int64_t cols, int64_t ld)
{
    if ((reinterpret_cast<uintptr_t>(C) & 15) || (ld * 2) % 16) return false;
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
    cuuint32_t box[2] = {16, 32};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, C, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_32B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

// C [rows, cols] bf16 (row pitch ld elements) for TMA stores of 32 x 32
// boxes with the 64-byte swizzle; elements beyond the extents are not written.
bool make_map_c32(CUtensorMap *m, void *C, int64_t rows, int64_t cols, int64_t ld)
{
    if ((reinterpret_cast<uintptr_t>(C) & 15) || (ld * 2) % 16) return false;
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, C, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

bool make_map_bf16(CUtensorMap *m, const void *ptr, int64_t rows, int64_t K, int64_t ld, int box_rows)
{
    return make_map(m, ptr, rows, K, ld, box_rows);
}

// Bytes [rows, width] row-major (fp8 or packed fp4 codes): boxes of 128 bytes
// x box_rows rows, 128-byte swizzle, out-of-range bytes read as zero.
bool make_map_u8(CUtensorMap *m, const void *ptr, int64_t rows, int64_t width, int box_rows)
{
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)width, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)width};
    cuuint32_t box[2] = {128, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(ptr), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Packed 4-bit weights as uint32 words [rows, K/8]; box 16 words (128 k) x
// box_rows rows with the 64-byte swizzle (16-byte piece c of row r lands at
// piece c ^ ((r / 2) % 4)), out-of-range words read as zero.
bool make_map_words16(CUtensorMap *m, const void *ptr, int64_t rows, int64_t K, int box_rows)
{
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)(K / 8), (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(K / 8) * 4};
    cuuint32_t box[2] = {16, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Packed 4-bit weights as uint32 words [rows, K/8]; box 32 words (256 k) x
// box_rows rows with the 128-byte swizzle (16-byte piece c of row r lands at
// piece c ^ (r % 8)), out-of-range words read as zero.
bool make_map_words(CUtensorMap *m, const void *ptr, int64_t rows, int64_t K, int box_rows)
{
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {(cuuint64_t)(K / 8), (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(K / 8) * 4};
    cuuint32_t box[2] = {32, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Packed 4-bit weights [rows, K/8] (uint32), K a multiple of 256, as the 3-D
// view [K / 256][rows][32 words]: a box of box_kb 256-k blocks x box_rows rows
// lands as box_kb consecutive make_map_words boxes (128-byte swizzle).
bool make_map_words_kblocks(CUtensorMap *m, const void *ptr, int64_t rows, int64_t K, int box_rows, int box_kb)
{
    if (K % 256) return false;
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {32, (cuuint64_t)rows, (cuuint64_t)(K / 256)};
    cuuint64_t strides[2] = {(cuuint64_t)(K / 8) * 4, 128};
    cuuint32_t box[3] = {32, (cuuint32_t)box_rows, (cuuint32_t)box_kb};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<void *>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Pipeline depth per tile width.  Skinny (decode) kernels come in a deep form
// (one CTA per SM, about 190 KB of shared memory) used when the grid fits in
// one wave, and a shallow form (two CTAs per SM, about 100 KB each) for grids
// of up to two CTAs per SM.  Prefill uses one CTA per SM.
int umma_stages(int bn, bool skinny, bool deep)
{
    if (!skinny) return bn <= 192 ? 5 : 4;
    if (deep) return bn <= 64 ? 8 : 6;
    return bn <= 16 ? 6 : bn <= 32 ? 5 : bn <= 64 ? 4 : 3;
}

// W4A16 skinny kernels: one CTA per SM; packed stages of 256 k (16 KB).
int umma_w4_stages(int bn) { return bn <= 32 ? 8 : bn <= 64 ? 6 : 5; }

namespace {
template <int BN, int STAGES, bool SWAP, int MINB, bool W4 = false>
int cluster_capacity_t(int cluster)
{
    using L = Layout<BN, STAGES, W4, SWAP && MINB == 1>;
    auto kern = k_umma<BN, STAGES, SWAP, MINB, W4, false>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM) != cudaSuccess)
        return -1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(cluster * 64), 1, 1);
    cfg.blockDim = dim3(threads_for(W4), 1, 1);
    cfg.dynamicSmemBytes = L::SMEM;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = (unsigned)cluster;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) return -1;
    return n;
}
}  // namespace

// Clusters of `cluster` CTAs of the skinny kernel that can be resident at
// once on the current device (cached per device); -1 if the query fails.
int umma_cluster_capacity(int bn, bool deep, int cluster, bool w4)
{
    static std::mutex mu;
    static int cache[64][5][3][9];
    static bool have[64][5][3][9];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cluster < 1 || cluster > 8) return -1;
    const int bi = bn <= 16 ? 0 : bn <= 32 ? 1 : bn <= 64 ? 2 : bn <= 128 ? 3 : 4;
    const int kind = w4 ? 2 : (deep ? 1 : 0);
    std::lock_guard<std::mutex> lk(mu);
    int &slot = cache[dev & 63][bi][kind][cluster];
    if (!have[dev & 63][bi][kind][cluster]) {
        int n = -1;
        if (w4) {
            switch (bi) {
            case 0: n = cluster_capacity_t<16, 8, true, 1, true>(cluster); break;
            case 1: n = cluster_capacity_t<32, 8, true, 1, true>(cluster); break;
            case 2: n = cluster_capacity_t<64, 6, true, 1, true>(cluster); break;
            case 3: n = cluster_capacity_t<128, 5, true, 1, true>(cluster); break;
            default: break;
            }
        } else if (deep) {
            switch (bi) {
            case 0: n = cluster_capacity_t<16, 8, true, 1>(cluster); break;
            case 1: n = cluster_capacity_t<32, 8, true, 1>(cluster); break;
            case 2: n = cluster_capacity_t<64, 8, true, 1>(cluster); break;
            case 3: n = cluster_capacity_t<128, 6, true, 1>(cluster); break;
            default: break;
            }
        } else {
            switch (bi) {
            case 0: n = cluster_capacity_t<16, 6, true, 2>(cluster); break;
            case 1: n = cluster_capacity_t<32, 5, true, 2>(cluster); break;
            case 2: n = cluster_capacity_t<64, 4, true, 2>(cluster); break;
            case 3: n = cluster_capacity_t<128, 3, true, 2>(cluster); break;
            default: break;
            }
        }
        slot = n;
        have[dev & 63][bi][kind][cluster] = n >= 0;
    }
    return slot;
}

int g_debug_stall = 0;

namespace {
// Activations [M, K] (K % 8 == 0) copied with every 8-k block reordered to
// k = 0, 4, 1, 5, 2, 6, 3, 7: the order in which the W4A16 kernel lays the
// dequantised weights along K.  One thread per 16-byte block.
__global__ void __launch_bounds__(256) k_permute_k8(const uint4 *__restrict__ in, uint4 *__restrict__ out,
                                                    int64_t blocks)
{
    ptx::pdl_wait();                 // the workspace may still be read by the previous kernel
    ptx::pdl_launch_dependents();
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < blocks;
         i += (int64_t)gridDim.x * blockDim.x) {
        const uint4 a = ld_ro_v4(reinterpret_cast<const uint16_t *>(in + i));   // (a0 a1)(a2 a3)(a4 a5)(a6 a7)
        uint4 b;
        b.x = __byte_perm(a.x, a.z, 0x5410);   // (a0, a4)
        b.y = __byte_perm(a.x, a.z, 0x7632);   // (a1, a5)
        b.z = __byte_perm(a.y, a.w, 0x5410);   // (a2, a6)
        b.w = __byte_perm(a.y, a.w, 0x7632);   // (a3, a7)
        out[i] = b;
    }
}

cudaError_t launch_permute_k8(const void *in, void *out, int64_t M, int64_t K, const LaunchCtx &c)
{
    const int64_t blocks = M * K / 8;
    int64_t grid = (blocks + 255) / 256;
    if (grid > (int64_t)c.sm_count * 4) grid = (int64_t)c.sm_count * 4;
    if (grid < 1) grid = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = c.stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_permute_k8, reinterpret_cast<const uint4 *>(in), reinterpret_cast<uint4 *>(out),
                              blocks);
}
}  // namespace

cudaError_t launch_umma_w4a16(const GemmArgs &a, const Plan &p, const LaunchCtx &c)
{
    // skinny only: X = packed weights [N, K/8], Y = activations [M, K] in the kernel's k order
    if (!c.act_copy) return cudaErrorInvalidValue;
    cudaError_t e = launch_permute_k8(a.A, c.act_copy, a.M, a.K, c);
    if (e != cudaSuccess) return e;
    CUtensorMap mx, my;
    if (!make_map_packed(&mx, a.B, a.N, a.K) || !make_map(&my, c.act_copy, a.M, a.K, a.K, p.bn))
        return cudaErrorInvalidValue;
    Sched s{};
    s.mode = p.mode;
    s.tiles_r = (int)((a.N + BM - 1) / BM);
    s.tiles_q = (int)((a.M + p.bn - 1) / p.bn);
    s.tiles = s.tiles_r * s.tiles_q;
    s.nk = (int)((a.K + 4 * BK - 1) / (4 * BK));   // 256-k stages
    s.grid = p.grid;
    s.group_r = p.group_r > 0 ? p.group_r : s.tiles_r;
    s.whole = 0;
    s.sk_grid = p.grid;
    s.units = (long long)s.tiles * s.nk;
    s.stall = g_debug_stall;
    s.split = p.split;
    W4Args w4{(const uint16_t *)a.scales, (const uint8_t *)a.zeros, (int)a.K, (int)(a.K / a.group), (int)a.group,
              a.group == 32 ? 5 : a.group == 64 ? 6 : 7};
    uint16_t *C = (uint16_t *)a.C;
    const int r = (int)a.N, q = (int)a.M;
    s.epi = GEMM_EPI_NONE;
    CUtensorMap mc;
    if (!cluster_store_map(&mc, s, p, C, a.N, a.M, a.ldc)) mc = mx;   // (then unused)
    switch (p.bn) {
    case 16: return launch_t<16, 8, true, 1, true>(mx, my, mc, C, r, q, a.ldc, s, c, w4);
    case 32: return launch_t<32, 8, true, 1, true>(mx, my, mc, C, r, q, a.ldc, s, c, w4);
    case 64: return launch_t<64, 6, true, 1, true>(mx, my, mc, C, r, q, a.ldc, s, c, w4);
    case 128: return launch_t<128, 5, true, 1, true>(mx, my, mc, C, r, q, a.ldc, s, c, w4);
    default: return cudaErrorInvalidValue;
    }
}

namespace {
template <bool FUSED>
cudaError_t launch_bf16_t(const CUtensorMap &mx, const CUtensorMap &my, const CUtensorMap &mc, uint16_t *C, int r,
                          int q, int64_t ldc, const Sched &s, const Plan &p, const LaunchCtx &c, bool swap)
{
    if (swap && p.ctas_per_sm == 1) {
        switch (p.bn) {
        case 16: return launch_t<16, 8, true, 1, false, FUSED>(mx, my, mc, C, r, q, ldc, s, c);
        case 32: return launch_t<32, 8, true, 1, false, FUSED>(mx, my, mc, C, r, q, ldc, s, c);
        case 64: return launch_t<64, 8, true, 1, false, FUSED>(mx, my, mc, C, r, q, ldc, s, c);
        case 128: return launch_t<128, 6, true, 1, false, FUSED>(mx, my, mc, C, r, q, ldc, s, c);
        default: return cudaErrorInvalidValue;
        }
    }
    if (swap) {
        switch (p.bn) {
        case 16: return launch_t<16, 6, true, 2, false, FUSED>(mx, my, mc, C, r, q, ldc, s, c);
        case 32: return launch_t<32, 5, true, 2, false, FUSED>(mx, my, mc, C, r, q, ldc, s, c);
        case 64: return launch_t<64, 4, true, 2, false, FUSED>(mx, my, mc, C, r, q, ldc, s, c);
        case 128: return launch_t<128, 3, true, 2, false, FUSED>(mx, my, mc, C, r, q, ldc, s, c);
        default: return cudaErrorInvalidValue;
        }
    }
    switch (p.bn) {
    case 256: return launch_t<256, 4, false, 1, false, FUSED>(mx, my, mc, C, r, q, ldc, s, c);
    case 224: return launch_t<224, 4, false, 1, false, FUSED>(mx, my, mc, C, r, q, ldc, s, c);
    case 192: return launch_t<192, 5, false, 1, false, FUSED>(mx, my, mc, C, r, q, ldc, s, c);
    case 176: return launch_t<176, 5, false, 1, false, FUSED>(mx, my, mc, C, r, q, ldc, s, c);
    default: return cudaErrorInvalidValue;
    }
}
}  // namespace

cudaError_t launch_umma_bf16(const GemmArgs &a, const Plan &p, const LaunchCtx &c)
{
    const bool swap = p.variant == GEMM_VARIANT_SKINNY;
    const bool pairs = a.epi == GEMM_EPI_SILU_MUL;
    const int64_t NW = pairs ? 2 * a.N : a.N;   // weight rows the kernel multiplies
    const void *X = swap ? a.B : a.A;
    const void *Y = swap ? a.A : a.B;
    const int64_t R = swap ? NW : a.M, Q = swap ? a.M : NW;
    const int64_t ldx = swap ? a.ldb : a.lda, ldy = swap ? a.lda : a.ldb;
    CUtensorMap mx, my;
    const int64_t QY = a.gends ? a.groups * a.N : Q;   // grouped: B stacks the experts' weights
    // One token tile (prefill kernel, M <= 128): the X box covers the token rows
    // only, rounded up to 16.  Boxes that are mostly out of range were slow
    // (M = 8, 176-row weight tiles: 42.5 us with 128-row boxes, 31.9 with 16);
    // the MMA's remaining A rows hold stale shared memory and produce C rows
    // that are never stored (row m of C depends on row m of A alone).
    const int xbox = !swap && !a.gends && R <= BM ? (int)((R + 15) / 16 * 16) : BM;
    const bool okx = swap && pairs ? make_map_pairs(&mx, X, a.N, a.K, ldx, BM / 2) : make_map(&mx, X, R, a.K, ldx, xbox);
    const bool oky = !swap && pairs ? make_map_pairs(&my, Y, a.N, a.K, ldy, p.bn / 2) : make_map(&my, Y, QY, a.K, ldy, p.bn);
    if (!okx || !oky) return cudaErrorInvalidValue;
    Sched s{};
    s.mode = p.mode;
    s.tiles_r = (int)((R + BM - 1) / BM);
    s.tiles_q = (int)((Q + p.bn - 1) / p.bn);
    s.tiles = s.tiles_r * s.tiles_q;
    s.nk = (int)((a.K + BK - 1) / BK);
    s.grid = p.grid;
    s.group_r = p.group_r > 0 ? p.group_r : s.tiles_r;
    s.whole = p.mode == 1 ? p.whole : 0;
    // (a caller may shrink the grid to fit a fixed workspace: every CTA sharing
    // the stream-K units must exist)
    s.sk_grid = p.mode == 1 && p.sk_grid > 0 ? std::min(p.sk_grid, p.grid) : p.grid;
    s.units = (long long)(s.tiles - s.whole) * s.nk;
    s.stall = g_debug_stall;
    s.epi = a.epi;
    s.pairs = pairs ? 1 : 0;
    s.bias = (const uint16_t *)a.bias;
    s.gends = a.gends;
    s.groups = (int)a.groups;
    s.gN = (int)a.N;
    if (a.gends && (swap || p.mode != 0 || p.bn != 256)) return cudaErrorInvalidValue;
    uint16_t *C = (uint16_t *)a.C;
    s.split = p.split;
    s.x_bytes = xbox * BK * 2;
    CUtensorMap mc;
    if (!cluster_store_map(&mc, s, p, C, R, Q, a.ldc)) mc = mx;   // (then unused)
    return a.epi != GEMM_EPI_NONE ? launch_bf16_t<true>(mx, my, mc, C, (int)R, (int)Q, a.ldc, s, p, c, swap)
                                  : launch_bf16_t<false>(mx, my, mc, C, (int)R, (int)Q, a.ldc, s, p, c, swap);
}

}  // namespace dbw
