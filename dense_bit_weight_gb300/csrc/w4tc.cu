// w4tc.cu -- W4A16 decode on the 5th-generation tensor core with the zero
// point and the scale applied once per quantisation group.
//
// The contraction is the W4A16 decode GEMM of the hk-dsl PyPI page
// ("Results", W4A16 decode GEMM (AWQ)): w[n,k] = (q[n,k] - z[n,g]) * s[n,g],
// g = k / group.  Within a group s and z are constants, so
//     sum_{k in g} w a = s * D_g + c * S_g,   c = -(128 + z) * s,
//     D_g = sum_{k in g} (128 + q) a,         S_g = sum_{k in g} a.
// 128 + q is exact in bf16 as (0x4300 | q): the MMA operand of a pair of
// weights costs one mask (and for three of four nibble pairs a shift), and no
// weight is ever rounded.  D_g is an fp32 MMA result of its own in tensor
// memory; s * D_g + c * S_g is added in fp32 per group (c is exact in fp32:
// an 8-bit scale times an integer below 144).  Integer inputs stay exact.
//
// Swap AB: the weight rows are the MMA's 128-row A side, read from tensor
// memory (tcgen05.mma ... [a_tmem]); the tokens (a tile of BN = 16, 32 or 64)
// are its N side, read from shared memory.
//
// Roles (one CTA per SM, 15 warps):
//   warp 0      TMA producer of the packed weights: one 128-row x 128-k stage
//               (16 words per row, 8 KB, 64-byte swizzle) per slot of a ring
//   warp 1      allocates (and at exit frees) the tensor memory
//   warps 2-5   epilogue: per group, read D_g (tcgen05.ld), release it, add
//               s D_g + c S_g to fp32 registers; at a segment's end store the
//               tile or its stream-K partial (deterministic fixup)
//   warp 6      TMA producer of the activations (the pre-pass's copy in the
//               0,4,1,5,2,6,3,7 order of each 8-k block): BN x 128 k per stage
//   warps 7-14  dequantisation and MMA issue: two warpgroups take the stages
//               alternately; a warp handles its 32 weight rows (its
//               tensor-memory lane quarter) for the whole 128-k stage, and one
//               warp of the group issues the stage's eight MMAs (K = 16) into
//               the accumulators of the stage's groups (a ring of ND).
//               The NXB tensor-memory stage buffers (6 or 4) are used in
//               turn, so each warpgroup can run NXB / 2 stages ahead.  Issuing from the warpgroups instead of a
//               dedicated MMA warp (measured: ~1000 cycles per stage there,
//               sharing its SMSP with dequantising warps, and a wake-up per
//               stage) keeps the MMA issue next to the data it waits for.
// The packed-weight and activation rings, the stage buffers and the
// accumulators are sized so that a slot is only ever used by the stages of
// one warpgroup: a waiter's previous use of a slot is then its own, and a
// parity wait can never mistake a phase two steps behind for a completed one.
// (Group 32 puts four groups in a stage, so it takes eight accumulators and
// token tiles of at most 32.)
//
// Tensor memory (512 columns): dequantised stage buffers b = 0..NXB-1 at
// columns 64 b (128 k each: column c of a buffer holds k pair c in the
// permuted order, bf16x2), accumulators d = 0..ND-1 after them, BN columns
// each.  The MMA issue is unrolled over the stage's eight k-steps (the group
// size is a template parameter).
//
// Schedule: stream-K over (weight tile, stage) units (sched.cuh), the
// deterministic last-arriver fixup summing the fp32 partials in k order.
//
// Every wait is bounded (waits.cuh): an expired wait raises the CTA's abort
// flag and the device error word; roles leave their loops, producers drain the
// copies they issued, the MMA warp its MMAs, and tensor memory is freed.
#include <cuda.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "sched.cuh"
#include "waits.cuh"

namespace dbw {
namespace {

constexpr int BM = kTileRows;   // weight rows per tile
constexpr int KST = 128;        // k per stage
constexpr int NWG = 2;          // dequantising warpgroups (stages alternate between them)
constexpr uint32_t kXCols = KST / 2;          // tensor-memory columns of one dequantised stage
constexpr int kEpiWarp0 = 2, kActWarp = 6, kDqWarp0 = 7;
constexpr int kThreads = (kDqWarp0 + 4 * NWG) * 32;
constexpr int kEpiThreads = 128;

// BN: token tile; LG: log2 of the quantisation group.
template <int BN, int LG>
struct TcLayout {
    static constexpr int NGS = KST >> LG;                   // groups per stage
    // per-group accumulators (a ring): a multiple of NWG x NGS, so stage gs's
    // accumulators are used only by the stages of its own warpgroup
    static constexpr int ND = LG == 5 ? 8 : 4;
    static constexpr int NXB = BN <= 16 || (BN == 32 && LG > 5) ? 6 : 4;   // dequantised stage buffers
    static constexpr uint32_t DCOL = NXB * kXCols;          // first accumulator column
    static constexpr int STAGES = BN <= 32 ? 12 : 8;        // packed-weight ring (8 KB per slot)
    static constexpr int AST = BN <= 32 ? 8 : 4;            // activation ring
    static constexpr int PK_BYTES = BM * KST / 2;           // 8 KB of packed words per stage
    static constexpr int A_BYTES = BN * KST * 2;            // two 64-k boxes of BN rows
    static constexpr int A_OFF = STAGES * PK_BYTES;
    static constexpr int BAR_OFF = A_OFF + AST * A_BYTES;
    static constexpr int NBARS = 2 * STAGES + 2 * AST + 2 * NXB + 2 * ND + NWG + 1;
    static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;
    static constexpr int SMEM = MISC_OFF + 16 + 1024;       // + slack to align the base
    static_assert(STAGES % NWG == 0 && AST % NWG == 0 && NXB % NWG == 0, "ring slots must map to one warpgroup");
    static_assert(DCOL + ND * BN <= 512, "tensor-memory map");
    static_assert(ND % (NWG * NGS) == 0, "a warpgroup's accumulators are its own");
    static_assert(A_BYTES % 1024 == 0, "activation boxes keep the 1024-byte swizzle alignment");
};

// A ring of n slots walked in steps of k <= n: slot and the parity of the
// slot's current use.
struct Ring {
    int slot;
    uint32_t phase;
    int n;
    __device__ __forceinline__ void adv(int k)
    {
        slot += k;
        if (slot >= n) {
            slot -= n;
            phase ^= 1u;
        }
    }
};

struct TcArgs {
    const uint16_t *scales;   // bf16 [N, G]
    const uint8_t *zeros;     // uint8 [N, G]
    const float *gsum;        // fp32 [G][TP]: S_g per token (the pre-pass)
    int G, TP;                // groups per row; tokens of the group sums (whole token tiles)
};

// The last contributor's sum of a split tile, stored as bf16.  Out of line:
// the epilogue's per-group accumulators are dead here, and keeping the fixup's
// loads in a frame of their own keeps the main loop free of spills.
template <int BN>
__device__ __noinline__ void fixup_store(const Sched &sched, const float *__restrict__ ws, int t, int row,
                                         uint16_t *__restrict__ C, int64_t ldc, int R, int Q, int n, int qb)
{
    streamk_fixup<BN, (BN <= 32 ? 8 : 4)>(sched, ws, t, row, [=](int c0, const float(&f)[16]) {
        store_chunk<true>(C, ldc, R, Q, n, qb + c0, f);
    });
}

// LG: log2 of the quantisation group (5, 6 or 7).
template <int BN, int LG>
__global__ void __launch_bounds__(kThreads, 1)
k_w4tc(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmA, uint16_t *__restrict__ C,
       int R, int Q, int64_t ldc, const __grid_constant__ Sched sched, const TcArgs w, float *__restrict__ ws,
       int *__restrict__ counters,
       int *__restrict__ d_error)
{
    using L = TcLayout<BN, LG>;
    constexpr int STAGES = L::STAGES, AST = L::AST, NXB = L::NXB, ND = L::ND;
    constexpr uint32_t kDCol = L::DCOL;
    constexpr int GROUP = 1 << LG;
    constexpr int NGS = L::NGS;      // groups per stage: 1, 2 or 4
    constexpr uint32_t IDESC = ptx::idesc_bf16_f32(BM, BN);
    extern __shared__ uint8_t tc_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(tc_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = ptx::smem_addr(smem);
    const uint32_t bar0 = sbase + (uint32_t)L::BAR_OFF;
    auto FULL = [&](int s) { return bar0 + 8u * s; };
    auto EMPTY = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto AFULL = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
    auto AEMPTY = [&](int a) { return bar0 + 8u * (2 * STAGES + AST + a); };
    auto XFULL = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 * AST + b); };
    auto XEMPTY = [&](int b) { return bar0 + 8u * (2 * STAGES + 2 * AST + NXB + b); };
    auto DFULL = [&](int d) { return bar0 + 8u * (2 * STAGES + 2 * AST + 2 * NXB + d); };
    auto DEMPTY = [&](int d) { return bar0 + 8u * (2 * STAGES + 2 * AST + 2 * NXB + ND + d); };
    auto DONE = [&](int u) { return bar0 + 8u * (2 * STAGES + 2 * AST + 2 * NXB + 2 * ND + u); };
    const uint32_t FIXB = bar0 + 8u * (2 * STAGES + 2 * AST + 2 * NXB + 2 * ND + NWG);   // epilogue warps' barrier
    uint32_t *misc = reinterpret_cast<uint32_t *>(smem + L::MISC_OFF);   // [0] tmem, [1] abort, [2] last flag
    volatile uint32_t *abort_flag = misc + 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(FULL(s), 1);
            ptx::mbar_init(EMPTY(s), 4);   // the four warps of the warpgroup that read it
        }
        for (int a = 0; a < AST; ++a) {
            ptx::mbar_init(AFULL(a), 1);
            ptx::mbar_init(AEMPTY(a), 1);
        }
        for (int b = 0; b < NXB; ++b) {
            ptx::mbar_init(XFULL(b), 4);
            ptx::mbar_init(XEMPTY(b), 1);
        }
        for (int d = 0; d < ND; ++d) {
            ptx::mbar_init(DFULL(d), 1);
            ptx::mbar_init(DEMPTY(d), kEpiThreads / 32);
        }
        for (int u = 0; u < NWG; ++u) ptx::mbar_init(DONE(u), 1);
        ptx::mbar_init(FIXB, kEpiThreads / 32);
        misc[1] = 0;
        misc[2] = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_addr(misc), 512);
        ptx::tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tmQ);
        ptx::prefetch_tmap(&tmA);
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = misc[0];
    ptx::pdl_launch_dependents();

    if (warp == 0 || warp == kActWarp) {
        // ------------------------------------------------------------ producers
        // The packed weights are not written by the preceding kernel (the
        // activation pre-pass), which waited for all earlier work before this
        // grid could start, so warp 0 needs no dependency wait.
        if (lane == 0) {
            const bool packed = warp == 0;
            if (!packed) ptx::pdl_wait();   // the activation copy
            const uint64_t pol = packed ? ptx::policy_evict_first() : ptx::policy_evict_last();
            Ring ring{0, 0u, packed ? STAGES : AST};
            int issued = 0;
            SegIter it(sched, blockIdx.x, sched.tiles);
            Segment seg;
            bool ok = true;
            while (ok && it.next(sched, seg)) {
                int tr, tq;
                tile_coords(sched, seg.tile, tr, tq);
                for (int kb = seg.kb0; kb < seg.kb1; ++kb, ring.adv(1)) {
                    const uint32_t full = packed ? FULL(ring.slot) : AFULL(ring.slot);
                    if (!wait_bar(packed ? EMPTY(ring.slot) : AEMPTY(ring.slot), ring.phase ^ 1u, abort_flag, d_error)) {
                        ok = false;
                        break;
                    }
                    if (sched.stall) continue;
                    if (packed) {
                        ptx::mbar_arrive_expect_tx(full, L::PK_BYTES);
                        ptx::tma_load_2d(sbase + ring.slot * L::PK_BYTES, &tmQ, full, kb * (KST / 8), tr * BM, pol);
                    } else {
                        ptx::mbar_arrive_expect_tx(full, L::A_BYTES);
                        const uint32_t dst = sbase + L::A_OFF + ring.slot * L::A_BYTES;
                        ptx::tma_load_2d(dst, &tmA, full, kb * KST, tq * BN, pol);
                        ptx::tma_load_2d(dst + BN * 128, &tmA, full, kb * KST + 64, tq * BN, pol);
                    }
                    ++issued;
                }
            }
            if (!ok) {   // every slot's most recent copy lands before exit
                for (int s2 = 0; s2 < ring.n; ++s2) {
                    if (issued <= s2) continue;
                    const int last = issued - 1 - ((issued - 1 - s2) % ring.n);
                    wait_bar_drain(packed ? FULL(s2) : AFULL(s2), (uint32_t)((last / ring.n) & 1));
                }
            }
        }
    } else if (warp >= kDqWarp0) {
        // ------------------------------------------------------------ dequantisation and MMA issue
        // Warpgroup u takes the stages u, u + NWG, ...; warp q4 (its
        // tensor-memory lane quarter) handles weight rows 32 q4 .. 32 q4 + 31,
        // lane l row r = 32 q4 + l.  A thread reads its row's 16 packed words
        // (four 16-byte pieces, conflict-free under the 64-byte swizzle),
        // releases the slot, forms the 64 bf16x2 columns 128 + q (column 4w + j
        // of word w holds nibbles j and j + 4: k pair j of the permuted 8-k
        // block) and stores them into the stage's buffer; every warp then
        // arrives on XFULL.  One warp of the group (the issuer; the two groups'
        // issuers sit on different SMSPs) waits for the other three, the
        // stage's activations and free accumulators, and issues the stage's
        // eight MMAs itself: a group's MMAs write accumulators no other group
        // writes, so no ordering between issuing warps is needed, and no
        // separate MMA warp has to be woken per stage.
        const int u = (warp - kDqWarp0) >> 2;
        const int q4 = warp & 3;
        const bool issuer = q4 == (u == 0 ? 1 : 3);
        const int r = 32 * q4 + lane;
        const uint32_t row_off = (uint32_t)(r * 64);
        const uint32_t sw = (uint32_t)((r >> 1) & 3);
        const uint32_t trow = tmem + ((uint32_t)(32 * q4) << 16);
        // rings at this group's first stage; every own stage advances them by NWG
        Ring pk{u, 0u, STAGES}, act{u, 0u, AST}, xb{u, 0u, NXB};
        uint32_t gc = (uint32_t)(u * NGS);   // this stage's first group (accumulator gc % ND)
        int cyc = 0;
        SegIter it(sched, blockIdx.x, sched.tiles);
        Segment seg;
        bool ok = true;
        while (ok && it.next(sched, seg)) {
            for (int kb = seg.kb0; kb < seg.kb1; ++kb) {
                const bool own = cyc == u;
                cyc = cyc + 1 == NWG ? 0 : cyc + 1;
                if (!own) continue;
                if (!wait_bar_warp(FULL(pk.slot), pk.phase, abort_flag, d_error)) {
                    ok = false;
                    break;
                }
                const uint32_t sp = sbase + pk.slot * L::PK_BYTES + row_off;
                uint4 wv[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) wv[c] = ptx::lds128(sp + ((((uint32_t)c) ^ sw) << 4));
                arrive_warp(EMPTY(pk.slot));   // the slot may be refilled
                const bool pxe = ptx::mbar_test_wait(XEMPTY(xb.slot), xb.phase ^ 1u);
                const uint32_t xa = trow + (uint32_t)xb.slot * kXCols;
#pragma unroll
                for (int h = 0; h < 2; ++h) {   // words 8h .. 8h + 7 -> columns 32h .. 32h + 31
                    uint32_t v[32];
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        const uint4 q = wv[2 * h + c];
                        const uint32_t words[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e)
#pragma unroll
                            for (int j = 0; j < 4; ++j)
                                v[16 * c + 4 * e + j] = ((words[e] >> (4 * j)) & 0x000F000Fu) | 0x43004300u;
                    }
                    if (h == 0) {
                        // the buffer's previous stage was issued NXB stages ago
                        if (!settle_warp(pxe, XEMPTY(xb.slot), xb.phase ^ 1u, abort_flag, d_error)) {
                            ok = false;
                            break;
                        }
                        ptx::tc_fence_after();
                    }
                    ptx::tmem_st32(xa + 32u * (uint32_t)h, v);
                }
                if (!ok) break;
                ptx::tmem_wait_st();
                ptx::tc_fence_before();   // the MMAs read these columns after XFULL
                arrive_warp(XFULL(xb.slot));
                if (issuer) {
                    bool go = wait_bar_warp(XFULL(xb.slot), xb.phase, abort_flag, d_error) &&
                              wait_bar_warp(AFULL(act.slot), act.phase, abort_flag, d_error);
#pragma unroll
                    for (int i = 0; i < NGS; ++i)
                        go = go && wait_bar_warp(DEMPTY((gc + i) % ND), (((gc + i) / ND) & 1u) ^ 1u, abort_flag, d_error);
                    if (!go) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t xm = tmem + (uint32_t)xb.slot * kXCols;
                    const uint32_t ab = sbase + L::A_OFF + act.slot * L::A_BYTES;
                    const uint64_t bd0 = ptx::sdesc_kmajor_sw128(ab), bd1 = ptx::sdesc_kmajor_sw128(ab + BN * 128);
#pragma unroll
                    for (int kk = 0; kk < KST / 16; ++kk) {   // 16 k per MMA; group kk * 16 >> LG of the stage
                        const int kp = 16 * kk;
                        const uint32_t d = (gc + (uint32_t)(kp >> LG)) % ND;
                        ptx::mma_bf16_ts_warp(tmem + kDCol + d * BN, xm + (uint32_t)(kp >> 1),
                                              (kp < 64 ? bd0 : bd1) + (uint64_t)(2 * ((kp & 63) >> 4)), IDESC,
                                              (kp & (GROUP - 1)) ? 1u : 0u);
                        if (((kp + 16) & (GROUP - 1)) == 0) ptx::mma_commit_warp(DFULL(d));
                    }
                    ptx::mma_commit_warp(XEMPTY(xb.slot));
                    ptx::mma_commit_warp(AEMPTY(act.slot));
                }
                pk.adv(NWG);
                act.adv(NWG);
                xb.adv(NWG);
                gc += (uint32_t)(NWG * NGS);
            }
        }
        if (issuer) {   // every MMA this warp issued retires before tensor memory is freed
            ptx::mma_commit_warp(DONE(u));
            wait_bar_drain(DONE(u), 0);
        }
    } else if (warp >= kEpiWarp0 && warp < kEpiWarp0 + 4) {
        // ------------------------------------------------------------ epilogue (warps 2-5)
        const int q4 = warp & 3;            // tensor-memory lane quarter this warp may read
        const int row = q4 * 32 + lane;     // accumulator row = weight row within the tile
        const int etid = threadIdx.x - 32 * kEpiWarp0;
        const uint32_t tl = tmem + ((uint32_t)(q4 * 32) << 16) + kDCol;
        ptx::pdl_wait();                    // the group sums; C, workspace and counters may be in use before
        uint32_t gc = 0, fphase = 0;
        SegIter it(sched, blockIdx.x, sched.tiles);
        Segment seg;
        bool ok = true;
        while (ok && it.next(sched, seg)) {
            int tr, tq;
            tile_coords(sched, seg.tile, tr, tq);
            const int n = tr * BM + row;
            const bool nv = n < R;
            const uint16_t *srow = w.scales + (int64_t)(nv ? n : 0) * w.G;
            const uint8_t *zrow = w.zeros + (int64_t)(nv ? n : 0) * w.G;
            const float *gsum = w.gsum + tq * BN;
            float acc[BN];
#pragma unroll
            for (int j = 0; j < BN; ++j) acc[j] = 0.f;
            const int g0 = seg.kb0 * NGS, g1 = seg.kb1 * NGS;
            // scale and zero of the next group, loaded one group ahead
            float sn = 0.f, cn = 0.f;
            auto load_sc = [&](int gi, float &sv, float &cv) {
                const bool v = nv && gi < w.G;
                const uint32_t sb = v ? (uint32_t)__ldg(srow + gi) : 0u;
                const uint32_t zb = v ? (uint32_t)__ldg(zrow + gi) : 0u;
                sv = __uint_as_float(sb << 16);
                cv = -__uint_as_float(0x43000000u | (zb << 16)) * sv;   // -(128 + z) s, exact
            };
            load_sc(g0, sn, cn);
            for (int gi = g0; gi < g1; ++gi, ++gc) {
                const int d = (int)(gc % ND);
                const float sv = sn, cv = cn;
                if (gi + 1 < g1) load_sc(gi + 1, sn, cn);
                if (!wait_bar_warp(DFULL(d), (gc / ND) & 1u, abort_flag, d_error)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const bool live = gi < w.G;   // warp-uniform: groups past K (a ragged last stage) add nothing
#pragma unroll
                for (int c = 0; c < BN; c += 16) {
                    uint32_t dv[16];
                    ptx::tmem_ld16(tl + (uint32_t)(d * BN + c), dv);
                    ptx::tmem_wait_ld();
                    if (c + 16 >= BN) {   // the accumulator may be overwritten once every column is read
                        ptx::tc_fence_before();
                        arrive_warp(DEMPTY(d));
                    }
                    if (live) {
                        const float4 *sg = reinterpret_cast<const float4 *>(gsum + (int64_t)gi * w.TP + c);
#pragma unroll
                        for (int j4 = 0; j4 < 4; ++j4) {
                            const float4 s4 = __ldg(sg + j4);
                            acc[c + 4 * j4 + 0] = fmaf(sv, __uint_as_float(dv[4 * j4 + 0]), fmaf(cv, s4.x, acc[c + 4 * j4 + 0]));
                            acc[c + 4 * j4 + 1] = fmaf(sv, __uint_as_float(dv[4 * j4 + 1]), fmaf(cv, s4.y, acc[c + 4 * j4 + 1]));
                            acc[c + 4 * j4 + 2] = fmaf(sv, __uint_as_float(dv[4 * j4 + 2]), fmaf(cv, s4.z, acc[c + 4 * j4 + 2]));
                            acc[c + 4 * j4 + 3] = fmaf(sv, __uint_as_float(dv[4 * j4 + 3]), fmaf(cv, s4.w, acc[c + 4 * j4 + 3]));
                        }
                    }
                }
            }
            if (!ok) break;
            const int qb = tq * BN;
            const bool whole = seg.kb0 == 0 && seg.kb1 == sched.nk;
            if (whole) {
#pragma unroll
                for (int c = 0; c < BN; c += 16) {
                    float f[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) f[j] = acc[c + j];
                    store_chunk<true>(C, ldc, R, Q, n, qb + c, f);
                }
                continue;
            }
            // stream-K partial: float4 columns, [column / 4][row], so a warp's store is 512 contiguous bytes
            float4 *part = reinterpret_cast<float4 *>(ws) + (int64_t)(blockIdx.x * 2 + seg.slot) * (BM * BN / 4);
#pragma unroll
            for (int c4 = 0; c4 < BN / 4; ++c4)
                __stcg(part + c4 * BM + row, make_float4(acc[4 * c4], acc[4 * c4 + 1], acc[4 * c4 + 2], acc[4 * c4 + 3]));
            const int t = seg.tile;
            const int c_first = cta_of_unit(sched, (long long)t * sched.nk);
            const int c_last = cta_of_unit(sched, (long long)(t + 1) * sched.nk - 1);
            __threadfence();
            if (!group_sync_warp(FIXB, fphase, abort_flag, d_error)) break;
            if (etid == 0) {
                const int old = atomicAdd(counters + t, 1);
                const bool last = old == c_last - c_first;
                if (last) counters[t] = 0;
                misc[2] = last ? 1u : 0u;
            }
            if (!group_sync_warp(FIXB, fphase, abort_flag, d_error)) break;
            if (!misc[2]) continue;
            __threadfence();
            fixup_store<BN>(sched, ws, t, row, C, ldc, R, Q, n, qb);
        }
    }

    // every warp converged before the CTA barrier
    __syncwarp();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
}

template <int BN, int LG>
cudaError_t launch_tc_t(const CUtensorMap &mq, const CUtensorMap &ma, uint16_t *C, int R, int Q, int64_t ldc,
                        const Sched &s, const TcArgs &w, const LaunchCtx &c)
{
    using L = TcLayout<BN, LG>;
    auto kern = k_w4tc<BN, LG>;
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
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = L::SMEM;
    cfg.stream = c.stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, mq, ma, C, R, Q, ldc, s, w, c.workspace, c.counters, c.d_error);
}

}  // namespace

int w4tc_stages(int bn) { return bn <= 32 ? TcLayout<16, 7>::STAGES : TcLayout<64, 7>::STAGES; }

cudaError_t launch_w4tc(const GemmArgs &a, const Plan &p, const LaunchCtx &c)
{
    if (!c.act_copy || !c.workspace || !c.counters) return cudaErrorInvalidValue;
    const int bn = p.bn;
    const int64_t tiles_q = (a.M + bn - 1) / bn;
    const int TP = (int)(tiles_q * bn);
    uint16_t *Ap = (uint16_t *)c.act_copy;
    float *S = reinterpret_cast<float *>(Ap + (a.M * a.K + 127) / 128 * 128);
    cudaError_t e = launch_w4_prep(a, c, Ap, S, TP);
    if (e != cudaSuccess) return e;
    CUtensorMap mq, ma;
    if (!make_map_words16(&mq, a.B, a.N, a.K, BM) || !make_map_bf16(&ma, Ap, a.M, a.K, a.K, bn))
        return cudaErrorInvalidValue;
    Sched s{};
    s.mode = 1;
    s.tiles_r = (int)((a.N + BM - 1) / BM);
    s.tiles_q = (int)tiles_q;
    s.tiles = s.tiles_r * s.tiles_q;
    s.nk = (int)((a.K + KST - 1) / KST);
    s.grid = p.grid;
    s.group_r = p.group_r > 0 ? p.group_r : s.tiles_r;
    s.whole = 0;
    s.sk_grid = p.grid;
    s.units = (long long)s.tiles * s.nk;
    s.stall = g_debug_stall;
    s.split = p.split;
    TcArgs w{(const uint16_t *)a.scales, (const uint8_t *)a.zeros, S, (int)(a.K / a.group), TP};
    uint16_t *C = (uint16_t *)a.C;
    const int lg = a.group == 32 ? 5 : a.group == 64 ? 6 : 7;
#define W4TC_CASE(BNV, LGV) \
    if (bn == BNV && lg == LGV) return launch_tc_t<BNV, LGV>(mq, ma, C, (int)a.N, (int)a.M, a.ldc, s, w, c);
    W4TC_CASE(16, 7) W4TC_CASE(16, 6) W4TC_CASE(16, 5)
    W4TC_CASE(32, 7) W4TC_CASE(32, 6) W4TC_CASE(32, 5)
    W4TC_CASE(64, 7) W4TC_CASE(64, 6)
#undef W4TC_CASE
    return cudaErrorInvalidValue;
}

}  // namespace dbw
