// umma2.cu -- the prefill GEMM on CTA pairs: tcgen05.mma.cta_group::2 with
// 256 x 256 output tiles, C = A . B^T (bf16 in, fp32 accumulation in tensor
// memory, bf16 out).
//
// The only Blackwell data point the pages give is a 256 x 256 output tile
// computed by a 256 x 256 x 16 MMA (HipKittens notes, Table 2, B200).  On
// sm_100-family hardware that MMA spans two SMs: the two CTAs of a cluster
// each hold half of the tile's A rows and half of its B rows in their own
// shared memory, and one instruction, issued by the pair's leader (cluster
// rank 0), multiplies the whole 256 x 256 x 16 block, each CTA's tensor
// memory receiving its own 128 rows of the accumulator.  Per CTA that is a
// 128 x 256 tile fed by 32 KB of operands per 64-k stage instead of the
// 48 KB a single-CTA 128 x 256 tile needs.
//
// Roles (320 threads per CTA, one CTA per SM, persistent over pair tiles):
//   warp 0      producer, in both CTAs: per stage the CTA's 128 rows of A and
//               its 128 rows of B (TMA, 128-byte swizzle), both copies
//               signalling the LEADER's full barrier (the .cta_group::2 form);
//               the leader's producer announces the bytes of both CTAs
//   warp 1      allocates the pair's tensor memory (both CTAs); in the leader
//               issues four MMAs (K = 16) per stage and commits the stage's
//               release and the accumulator's completion to the barriers of
//               both CTAs (multicast)
//   warps 2-9   epilogue, in both CTAs: two warps per quarter of the CTA's
//               128 accumulator rows (a warp reads only its quarter of the
//               tensor memory lanes), each taking 128 of the 256 columns ->
//               bf16 -> C through TMA stores; each warp then releases the
//               accumulator on the leader's barrier (sixteen arrivals)
// Two accumulators of 256 columns let the epilogue of one tile overlap the
// MMAs of the next.  Schedule (sched.cuh, the pairs as its CTAs): whole tiles
// round-robin, or stream-K ranges of (tile, k-block) units when whole tiles
// would leave the last wave of pairs mostly idle; a split tile's partials are
// kept per CTA half (each CTA its 128 rows) and summed in k order by the last
// contributor.  Every wait is bounded (waits.cuh); a cluster barrier
// before exit keeps either CTA from leaving while its partner may still
// signal its barriers or read its shared memory.
#include <cuda.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "frag.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "sched.cuh"
#include "waits.cuh"

namespace dbw {
namespace {

constexpr int BMC = kTileRows;      // A rows per CTA (256 per pair)
constexpr int BN = 256;             // B rows per pair tile (128 per CTA)
constexpr int BNC = BN / 2;
constexpr int BK = 64;
constexpr int STAGES = 6;
constexpr int A_BYTES = BMC * BK * 2;    // 16 KB
constexpr int B_BYTES = BNC * BK * 2;    // 16 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int kEpiWarps = 8;                       // warps 2-9
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int EPI_OFF = STAGES * STAGE_BYTES;      // the epilogue warps' staging boxes for C
constexpr int EPI_BOX_BYTES = 32 * 64;             // 32 rows x 32 bf16 columns
constexpr int EPI_WARP_BYTES = 2 * EPI_BOX_BYTES;  // two boxes per warp (double buffered)
constexpr int BAR_OFF = EPI_OFF + kEpiWarps * EPI_WARP_BYTES;
constexpr int FIX_SLOTS = STAGES;                  // staged fixup: 16 KB slots per column half
constexpr int FIX_SLOT_BYTES = STAGES * STAGE_BYTES / (2 * FIX_SLOTS);
constexpr int NBARS = 2 * STAGES + 4 + 1 + 3 + 2 * FIX_SLOTS;
constexpr int MISC_OFF = BAR_OFF + NBARS * 8;
constexpr int GRP_OFF = MISC_OFF + 16;             // grouped GEMM: expert row ends, m-tile prefix
constexpr int GRP_BYTES = 4 * (2 * kPairMaxExperts + 1);
constexpr int SMEM = GRP_OFF + GRP_BYTES + 1024;

__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// The pair's MMA (M = 256 over both CTAs), from one elected lane of a converged warp.
__device__ __forceinline__ void mma_pair_warp(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                              uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on the barrier at this shared-memory offset in both CTAs of the pair
// once the MMAs issued so far have completed.
__device__ __forceinline__ void commit_pair_warp(uint32_t bar)
{
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n\t}" ::"r"(
            bar),
        "h"((uint16_t)3)
        : "memory");
}

// 2-D tile load into this CTA's shared memory, completion counted on the
// barrier `bar_cluster` (a shared::cluster address: the leader's).
__device__ __forceinline__ void tma_load_pair(uint32_t dst, const CUtensorMap *m, uint32_t bar_cluster, int32_t c0,
                                              int32_t c1, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(bar_cluster), "r"(c0), "r"(c1), "l"(policy)
        : "memory");
}

// 3-D tile load (the (gate, up) row-pair view of a fused gate/up weight) into
// this CTA's shared memory, completion counted on the leader's barrier.
__device__ __forceinline__ void tma_load_pair_3d(uint32_t dst, const CUtensorMap *m, uint32_t bar_cluster, int32_t c0,
                                                 int32_t c1, int32_t c2, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(bar_cluster), "r"(c0), "r"(c1), "r"(c2), "l"(policy)
        : "memory");
}

// Arrive on this CTA's barrier once the MMAs issued so far have completed.
__device__ __forceinline__ void commit_local_warp(uint32_t bar)
{
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
        : "memory");
}

__device__ __forceinline__ void arrive_remote(uint32_t bar_cluster)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}

__device__ __forceinline__ void bulk_wait_read1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }

// bf16 store of W (32 or 16) columns of this warp's 32 accumulator rows
// (row r0 + lane held by each lane): the lanes write a 32 x W box into one of
// the warp's two staging boxes in shared memory and lane 0 hands it to the
// TMA engine, which writes the rows of C (clipping rows >= M and columns >=
// N), while the warp goes on with the next box.  The box uses the swizzle of
// its C map (64-byte rows: chunk j of row x at j ^ ((x / 2) % 4); 32-byte rows:
// j ^ ((x / 4) % 2)), so the lanes' writes spread over all banks.  Before a box
// is refilled, the store issued from it two boxes earlier has finished reading it.
template <int W>
__device__ __forceinline__ void store_box(const CUtensorMap *tmC, int M, int N, int r0, int q0, const float (&f)[W],
                                          uint32_t wbuf, int &sel, int lane)
{
    static_assert(W == 32 || W == 16, "boxes of 32 or 16 columns");
    if (r0 >= M || q0 >= N) return;   // the box lies wholly outside C
    const uint32_t box = wbuf + (uint32_t)(sel * EPI_BOX_BYTES);
    if (lane == 0) bulk_wait_read1();
    __syncwarp();
    const uint32_t sw = W == 32 ? (uint32_t)((lane >> 1) & 3) : (uint32_t)((lane >> 2) & 1);
#pragma unroll
    for (int j = 0; j < W / 8; ++j) {
        uint4 w;
        w.x = pack_bf16x2_rn(f[8 * j], f[8 * j + 1]);
        w.y = pack_bf16x2_rn(f[8 * j + 2], f[8 * j + 3]);
        w.z = pack_bf16x2_rn(f[8 * j + 4], f[8 * j + 5]);
        w.w = pack_bf16x2_rn(f[8 * j + 6], f[8 * j + 7]);
        ptx::sts128(box + (uint32_t)(lane * (2 * W)) + (((uint32_t)j ^ sw) << 4), w);
    }
    ptx::fence_proxy_async_smem();   // the box is read by the TMA engine
    __syncwarp();
    if (lane == 0) {
        ptx::tma_store_2d(tmC, box, q0, r0);
        ptx::bulk_commit_group();
    }
    sel ^= 1;
}

// The epilogue of 32 accumulator columns (c0 .. c0 + 31 of the tile, whose
// first output column is qb): plain or bias (+ activation) results go out as
// a 32-column box; with (gate, up) row pairs the columns alternate gate and
// up, and silu(gate) * up gives 16 output columns (qb + c0 / 2 ...).
template <bool PAIRS, bool GRP>
__device__ __forceinline__ void emit_cols(const CUtensorMap *tmC, const Sched &sched, int M, int N, int r0, int qb,
                                          int c0, float (&f)[32], uint32_t wbuf, int &sel, int lane, int rlim,
                                          uint16_t *__restrict__ Cg, int64_t ldc)
{
    if constexpr (GRP) {
        // an expert's last rows: the box would cross into the next expert's
        // rows of C, so this lane stores its own row (below rlim) directly
        if (r0 + 32 > rlim) {
            const int r = r0 + lane, q0 = qb + c0;
            if (r < rlim && q0 < N) {
                uint16_t *dst = Cg + (int64_t)r * ldc + q0;
                if (q0 + 32 <= N) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        uint4 w;
                        w.x = pack_bf16x2_rn(f[8 * j], f[8 * j + 1]);
                        w.y = pack_bf16x2_rn(f[8 * j + 2], f[8 * j + 3]);
                        w.z = pack_bf16x2_rn(f[8 * j + 4], f[8 * j + 5]);
                        w.w = pack_bf16x2_rn(f[8 * j + 6], f[8 * j + 7]);
                        reinterpret_cast<uint4 *>(dst)[j] = w;
                    }
                } else {
                    for (int j = 0; j < 32 && q0 + j < N; ++j) dst[j] = f32_to_bf16_rn(f[j]);
                }
            }
            return;
        }
    }
    if constexpr (PAIRS) {
        float o[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) o[j] = silu_mul(f[2 * j], f[2 * j + 1]);
        store_box<16>(tmC, M, N, r0, qb + c0 / 2, o, wbuf, sel, lane);
    } else {
        if (epi_has_bias(sched.epi)) {
            const int q0 = qb + c0;
            const uint16_t *bp = sched.bias + q0;
            if (q0 + 32 <= N && (reinterpret_cast<uintptr_t>(bp) & 15) == 0) {   // four 16-byte loads
#pragma unroll
                for (int j8 = 0; j8 < 4; ++j8) {
                    const uint4 w = ld_ro_v4(bp + 8 * j8);
                    const uint32_t h[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        f[8 * j8 + 2 * e] = bias_act(f[8 * j8 + 2 * e], bf16lo(h[e]), sched.epi);
                        f[8 * j8 + 2 * e + 1] = bias_act(f[8 * j8 + 2 * e + 1], bf16hi(h[e]), sched.epi);
                    }
                }
            } else {   // (a bias only 2-byte aligned, or the columns past N)
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float b = q0 + j < N ? bf16lo((uint32_t)__ldg(bp + j)) : 0.f;
                    f[j] = bias_act(f[j], b, sched.epi);
                }
            }
        }
        store_box<32>(tmC, M, N, r0, qb + c0, f, wbuf, sel, lane);
    }
}

// Stream-K fixup with plain loads (a split tile that is not this CTA's final
// segment, so the operand ring is busy): this warp's 128 columns, 32 at a
// time, the partials of the contributors in increasing order; the same sums,
// in the same order, as staged_fixup.  emit(c0, f) takes 32 columns.
template <typename Emit>
__device__ __forceinline__ void direct_fixup(const Sched &sched, const float *__restrict__ ws, int t, int row,
                                             int col0, Emit &emit)
{
    const int c_first = cta_of_unit(sched, (long long)t * sched.nk);
    const int c_last = cta_of_unit(sched, (long long)(t + 1) * sched.nk - 1);
    const float4 *wsv = reinterpret_cast<const float4 *>(ws);
#pragma unroll 1
    for (int cb = col0 / 4; cb < (col0 + BN / 2) / 4; cb += 8) {
        float4 a4[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) a4[j] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
        for (int cta = c_first; cta <= c_last; ++cta) {
            const int slot = (int)(range_begin(sched, cta) / sched.nk) == t ? 0 : 1;
            const float4 *p = wsv + (int64_t)(cta * 2 + slot) * (BMC * BN / 4) + (int64_t)cb * BMC + row;
            float4 v[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) v[j] = __ldcg(p + j * BMC);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                a4[j].x += v[j].x;
                a4[j].y += v[j].y;
                a4[j].z += v[j].z;
                a4[j].w += v[j].w;
            }
        }
        float f[32];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            f[4 * u] = a4[u].x;
            f[4 * u + 1] = a4[u].y;
            f[4 * u + 2] = a4[u].z;
            f[4 * u + 3] = a4[u].w;
        }
        emit(cb * 4, f);
    }
}

// Stream-K fixup of tile t by its last contributor, when the tile is this
// CTA's final segment: every MMA of the pair has then completed and no copy
// is in flight, so the operand ring stages the partials.  Each column half
// (four warps) has FIX_SLOTS slots of 16 KB and its own barriers; its chunk i
// (32 columns x 128 rows of contributor c_first + i % nc, column batch
// i / nc of the half) arrives by one bulk copy into slot i % FIX_SLOTS, all
// slots in flight at once, where plain loads would keep only a few KB per
// warp in flight and wait out the L2 latency many times.  Sums run over the
// contributors in increasing order, the same arithmetic as direct_fixup, so
// the bits do not depend on which path ran.  emit(c0, f) takes 32 columns.
// Returns false on a timeout or abort, after waiting (bounded) for the copies
// still in flight.
template <typename Emit>
__device__ __noinline__ bool staged_fixup(const Sched &sched, const float *__restrict__ ws, int t, int row, int half,
                                          bool issuer, const uint8_t *ring, uint32_t ring_s, uint32_t stg0,
                                          uint32_t hbar, uint32_t &hphase, volatile uint32_t *abort_flag,
                                          int *d_error, Emit &emit)
{
    constexpr int CHUNK_F4 = 8 * BMC;                   // 8 float4 columns of 128 rows
    constexpr uint32_t CHUNK_BYTES = CHUNK_F4 * 16;     // 16 KB, one slot
    static_assert(CHUNK_BYTES == (uint32_t)FIX_SLOT_BYTES, "a partial chunk fills one slot");
    const int c_first = cta_of_unit(sched, (long long)t * sched.nk);
    const int c_last = cta_of_unit(sched, (long long)(t + 1) * sched.nk - 1);
    const int nc = c_last - c_first + 1;
    constexpr int BATCHES = BN / 2 / 32;                // column batches of a half
    const int chunks = BATCHES * nc;
    const float4 *wsv = reinterpret_cast<const float4 *>(ws);
    auto issue = [&](int i) {
        const int cta = c_first + i % nc;
        const int slot = (int)(range_begin(sched, cta) / sched.nk) == t ? 0 : 1;
        const int cb = half * (BN / 8) + (i / nc) * 8;   // first float4 column of the batch
        const float4 *src = wsv + (int64_t)(cta * 2 + slot) * (BMC * BN / 4) + (int64_t)cb * BMC;
        const uint32_t bar = stg0 + 8u * (i % FIX_SLOTS);
        ptx::mbar_arrive_expect_tx(bar, CHUNK_BYTES);
        bulk_load(ring_s + (uint32_t)((i % FIX_SLOTS) * FIX_SLOT_BYTES), src, CHUNK_BYTES, bar);
    };
    int issued = 0;
    if (issuer) {
        // the partials were written by other threads' plain stores (released
        // through the tile counter); order them before the bulk copies read them
        asm volatile("fence.proxy.async.global;" ::: "memory");
        for (; issued < chunks && issued < FIX_SLOTS; ++issued) issue(issued);
    }
    bool ok = true;
    int i = 0;
    float4 a4[8];
    for (; i < chunks; ++i) {
        const int b = i % FIX_SLOTS;
        if (i % nc == 0) {
#pragma unroll
            for (int j = 0; j < 8; ++j) a4[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        if (!wait_bar_warp(stg0 + 8u * b, (uint32_t)(i / FIX_SLOTS) & 1u, abort_flag, d_error)) {
            ok = false;
            break;
        }
        const float4 *buf = reinterpret_cast<const float4 *>(ring + b * FIX_SLOT_BYTES);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float4 v = buf[j * BMC + row];
            a4[j].x += v.x;
            a4[j].y += v.y;
            a4[j].z += v.z;
            a4[j].w += v.w;
        }
        if (i + FIX_SLOTS < chunks) {
            // every warp of this half has read slot b: refill it
            if (!group_sync_warp(hbar, hphase, abort_flag, d_error)) {
                ok = false;
                ++i;
                break;
            }
            if (issuer) issue(issued++);
        }
        if (i % nc == nc - 1) {
            float f[32];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                f[4 * u] = a4[u].x;
                f[4 * u + 1] = a4[u].y;
                f[4 * u + 2] = a4[u].z;
                f[4 * u + 3] = a4[u].w;
            }
            emit(half * (BN / 2) + (i / nc) * 32, f);
        }
    }
    if (!ok && issuer) {
        // copies issued beyond the last one waited for are still landing
        for (int k = i; k < issued; ++k) wait_bar_drain(stg0 + 8u * (k % FIX_SLOTS), (uint32_t)(k / FIX_SLOTS) & 1u);
    }
    return ok;
}

template <bool PAIRS, bool GRP>
__global__ void __launch_bounds__(kThreads, 1)
k_umma_pair(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
            const __grid_constant__ CUtensorMap tmC, uint16_t *__restrict__ Cg, int64_t ldc, int M, int N,
            const __grid_constant__ Sched sched,
            float *__restrict__ ws,
            int *__restrict__ counters, int *__restrict__ d_error)
{
    constexpr uint32_t IDESC = ptx::idesc_bf16_f32(2 * BMC, BN);
    extern __shared__ uint8_t pair_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(pair_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = ptx::smem_addr(smem);
    const uint32_t bar0 = sbase + (uint32_t)BAR_OFF;
    auto FULL = [&](int s) { return bar0 + 8u * s; };
    auto EMPTY = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto TFULL = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
    auto TEMPTY = [&](int a) { return bar0 + 8u * (2 * STAGES + 2 + a); };
    const uint32_t DONE = bar0 + 8u * (2 * STAGES + 4);
    const uint32_t FIXB = bar0 + 8u * (2 * STAGES + 5);   // this CTA's epilogue warps (stream-K counter)
    const uint32_t HALFB = bar0 + 8u * (2 * STAGES + 6);  // [2]: the four warps of a column half
    const uint32_t STG0 = bar0 + 8u * (2 * STAGES + 8);   // [2][FIX_SLOTS]: partials staged for the fixup
    uint32_t *misc = reinterpret_cast<uint32_t *>(smem + MISC_OFF);   // [0] tmem, [1] abort, [2] last flag
    volatile uint32_t *abort_flag = misc + 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = ptx::cluster_ctarank();
    const bool leader = rank == 0;
    const int pair = (int)(blockIdx.x >> 1);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(FULL(s), 1);    // the leader's producer; both CTAs' copies count their bytes
            ptx::mbar_init(EMPTY(s), 1);   // the leader's multicast commit
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(TFULL(a), 1);
            ptx::mbar_init(TEMPTY(a), 2 * kEpiWarps);   // (used in the leader) both CTAs' epilogue warps
        }
        ptx::mbar_init(DONE, 1);
        ptx::mbar_init(FIXB, kEpiWarps);
        for (int h = 0; h < 2; ++h) ptx::mbar_init(HALFB + 8u * h, kEpiWarps / 2);
        for (int b = 0; b < 2 * FIX_SLOTS; ++b) ptx::mbar_init(STG0 + 8u * b, 1);
        misc[1] = 0;
        misc[2] = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(ptx::smem_addr(misc), 512);
        tmem_relinquish_pair();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tmA);
        ptx::prefetch_tmap(&tmB);
        ptx::prefetch_tmap(&tmC);
    }
    ptx::tc_fence_before();
    // both CTAs' barriers are initialised before any copy or commit signals them
    ptx::cluster_arrive_release();
    ptx::cluster_wait();
    __syncwarp();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = misc[0];

    // Grouped GEMM: expert g owns the token rows [end[g-1], end[g]) of A and C
    // and multiplies them by its weight rows g*gN .. g*gN + gN - 1 of B.  The
    // row ends come from the previous kernel (a router), so every thread waits
    // for them; warp 0 of each CTA clamps them into a non-decreasing sequence
    // within [0, M] and writes the exclusive prefix of the experts' 256-row
    // m-tile counts; expert g then owns the pair tiles from gpre[g] * tiles_q,
    // m-tile fastest, and an expert with no rows owns none.
    int *gend = reinterpret_cast<int *>(smem + GRP_OFF);
    int *gpre = gend + kPairMaxExperts;
    int ntiles = sched.tiles;
    if constexpr (GRP) {
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
            int prev = min(before, M), mt = 0;
            run = before;
            for (int g = g0; g < g1; ++g) {
                run = max(run, __ldg(sched.gends + g));
                const int e = min(run, M);
                gend[g] = e;
                mt += (e - prev + 2 * BMC - 1) / (2 * BMC);
                prev = e;
            }
            int base = mt;                   // exclusive sum-scan of the m-tile counts
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, base, o);
                if (lane >= o) base += v;
            }
            if (lane == 31) gpre[G] = base;
            base -= mt;
            prev = min(before, M);
            for (int g = g0; g < g1; ++g) {
                gpre[g] = base;
                base += (gend[g] - (g == g0 ? prev : gend[g - 1]) + 2 * BMC - 1) / (2 * BMC);
            }
        }
        __syncthreads();
        ntiles = gpre[sched.groups] * sched.tiles_q;
    }
    // pair tile t -> A rows from xrow (this CTA's half at xrow + 128 rank), B
    // rows from yrow, C rows below rlim, the first output column qb
    auto geo = [&](int t, int &xrow, int &yrow, int &rlim, int &qb) {
        if constexpr (GRP) {
            const int mt = t / sched.tiles_q;   // expert g owns tiles [gpre[g], gpre[g + 1]) * tiles_q
            int lo = 0, hi = sched.groups;      // the expert: largest lo < G with gpre[lo] <= mt
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (gpre[mid] <= mt) lo = mid;
                else hi = mid;
            }
            // within the expert, m-tiles vary fastest: the pairs that read one
            // weight tile run side by side, so it comes from DRAM once
            const int nm = gpre[lo + 1] - gpre[lo];
            const int local = t - gpre[lo] * sched.tiles_q;
            const int tqe = local / nm, mte = local - tqe * nm;
            xrow = (lo > 0 ? gend[lo - 1] : 0) + mte * (2 * BMC);
            rlim = gend[lo];
            yrow = lo * sched.gN + tqe * BN;
            qb = tqe * BN;
        } else {
            int tm, tn;
            tile_coords(sched, t, tm, tn);
            xrow = tm * (2 * BMC);
            yrow = tn * BN;
            rlim = M;
            qb = tn * (PAIRS ? BN / 2 : BN);   // a tile of (gate, up) row pairs has BN / 2 output columns
        }
    };
    ptx::pdl_launch_dependents();

    if (warp == 0) {
        // ------------------------------------------------------------ producer (both CTAs)
        if (lane == 0) {
            const uint64_t pol_a = ptx::policy_evict_last();
            const uint64_t pol_b = ptx::policy_evict_last();
            ptx::pdl_wait();
            int stage = 0, issued = 0;
            uint32_t phase = 0;
            bool ok = true;
            SegIter it(sched, pair, ntiles);
            Segment seg;
            while (ok && it.next(sched, seg)) {
                int xrow, yrow, rlim, qb;
                geo(seg.tile, xrow, yrow, rlim, qb);
                (void)rlim;
                for (int kb = seg.kb0; kb < seg.kb1; ++kb) {
                    if (!wait_bar(EMPTY(stage), phase ^ 1u, abort_flag, d_error)) {
                        ok = false;
                        break;
                    }
                    if (!sched.stall) {
                        const uint32_t full = ptx::map_cluster(FULL(stage), 0u);   // the leader's barrier
                        if (leader) ptx::mbar_arrive_expect_tx(FULL(stage), 2u * STAGE_BYTES);
                        const uint32_t st = sbase + (uint32_t)(stage * STAGE_BYTES);
                        tma_load_pair(st, &tmA, full, kb * BK, xrow + (int)rank * BMC, pol_a);
                        if (PAIRS)   // (gate, up) row pairs: 64 pairs per CTA
                            tma_load_pair_3d(st + A_BYTES, &tmB, full, kb * BK, 0, yrow / 2 + (int)rank * (BNC / 2),
                                             pol_b);
                        else
                            tma_load_pair(st + A_BYTES, &tmB, full, kb * BK, yrow + (int)rank * BNC, pol_b);
                        ++issued;
                    }
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            (void)issued;
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (leader)
        if (leader) {
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            SegIter it(sched, pair, ntiles);
            Segment seg;
            while (ok && it.next(sched, seg)) {
                if (!wait_bar_warp(TEMPTY(acc), acc_phase ^ 1u, abort_flag, d_error)) break;
                ptx::tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(acc * BN);
                for (int kb = seg.kb0; kb < seg.kb1; ++kb) {
                    if (!wait_bar_warp(FULL(stage), phase, abort_flag, d_error)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t st = sbase + (uint32_t)(stage * STAGE_BYTES);
                    const uint64_t ad = ptx::sdesc_kmajor_sw128(st), bd = ptx::sdesc_kmajor_sw128(st + A_BYTES);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k)
                        mma_pair_warp(d, ad + 2u * k, bd + 2u * k, IDESC, (kb > seg.kb0 || k > 0) ? 1u : 0u);
                    commit_pair_warp(EMPTY(stage));
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                commit_pair_warp(TFULL(acc));
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            commit_local_warp(DONE);   // every issued MMA retires before tensor memory is freed
            wait_bar_drain(DONE, 0);
        }
    } else {
        // ------------------------------------------------------------ epilogue (both CTAs)
        const int q4 = warp & 3;                 // tensor memory lane quarter this warp may read
        const int row = q4 * 32 + lane;
        const int half = (warp - 2) >> 2;        // columns [128 half, 128 half + 128)
        const int col0 = half * (BN / 2);
        ptx::pdl_wait();
        const uint32_t temp_leader0 = ptx::map_cluster(TEMPTY(0), 0u);
        const uint32_t temp_leader1 = ptx::map_cluster(TEMPTY(1), 0u);
        int acc = 0;
        uint32_t acc_phase = 0, fphase = 0, hphase = 0;
        const int etid = threadIdx.x - 64;
        const uint32_t wbuf = sbase + (uint32_t)(EPI_OFF + (warp - 2) * EPI_WARP_BYTES);
        int sel = 0;   // this warp's staging box for the next C store
        // stream-K: each CTA keeps its own half-tile partials and counters
        // (rank r's region), and the pairs act as the schedule's CTAs
        float *wsr = ws + (size_t)rank * ((size_t)sched.sk_grid * 2 * BMC * BN);
        int *cnt = counters + (size_t)rank * sched.tiles;
        SegIter it(sched, pair, ntiles);
        Segment seg;
        while (it.next(sched, seg)) {
            if (!wait_bar_warp(TFULL(acc), acc_phase, abort_flag, d_error)) break;
            ptx::tc_fence_after();
            int xrow, yrow, rlim, qb;
            geo(seg.tile, xrow, yrow, rlim, qb);
            const int r0 = xrow + (int)rank * BMC + q4 * 32;
            const uint32_t taddr = tmem + ((uint32_t)(q4 * 32) << 16) + (uint32_t)(acc * BN);
            const bool whole = seg.kb0 == 0 && seg.kb1 == sched.nk;
            float4 *part = reinterpret_cast<float4 *>(wsr) + (int64_t)(pair * 2 + seg.slot) * (BMC * BN / 4);
#pragma unroll 1
            for (int c = col0; c < col0 + BN / 2; c += 32) {
                uint32_t v[16], v2[16];
                __syncwarp();
                ptx::tmem_ld16(taddr + (uint32_t)c, v);
                ptx::tmem_ld16(taddr + (uint32_t)(c + 16), v2);
                ptx::tmem_wait_ld();
                float f[32];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    f[j] = __uint_as_float(v[j]);
                    f[16 + j] = __uint_as_float(v2[j]);
                }
                if (whole) {
                    emit_cols<PAIRS, GRP>(&tmC, sched, M, N, r0, qb, c, f, wbuf, sel, lane, rlim, Cg, ldc);
                } else {
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        __stcg(part + (c / 4 + u) * BMC + row, make_float4(f[4 * u], f[4 * u + 1], f[4 * u + 2], f[4 * u + 3]));
                }
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) arrive_remote(acc == 0 ? temp_leader0 : temp_leader1);
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
            if (whole) continue;
            // the last contributor (pair) of this half tile sums the partials in k order
            const int t = seg.tile;
            const int c_first = cta_of_unit(sched, (long long)t * sched.nk);
            const int c_last = cta_of_unit(sched, (long long)(t + 1) * sched.nk - 1);
            __threadfence();
            if (!group_sync_warp(FIXB, fphase, abort_flag, d_error)) break;
            if (etid == 0) {
                const int old = atomicAdd(cnt + t, 1);
                const bool last = old == c_last - c_first;
                if (last) cnt[t] = 0;
                misc[2] = last ? 1u : 0u;
            }
            if (!group_sync_warp(FIXB, fphase, abort_flag, d_error)) break;
            if (!misc[2]) continue;
            __threadfence();
            auto emit32 = [&](int c0, const float(&f)[32]) {
                float g[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) g[j] = f[j];
                emit_cols<PAIRS, GRP>(&tmC, sched, M, N, r0, qb, c0, g, wbuf, sel, lane, rlim, Cg, ldc);
            };
            SegIter peek = it;
            Segment after;
            if (peek.next(sched, after)) {
                direct_fixup(sched, wsr, t, row, col0, emit32);
            } else if (!staged_fixup(sched, wsr, t, row, half, (warp & 3) == 2 && lane == 0,
                                     smem + half * (FIX_SLOTS * FIX_SLOT_BYTES),
                                     sbase + (uint32_t)(half * (FIX_SLOTS * FIX_SLOT_BYTES)),
                                     STG0 + 8u * (uint32_t)(half * FIX_SLOTS), HALFB + 8u * (uint32_t)half, hphase,
                                     abort_flag, d_error, emit32)) {
                break;
            }
        }
    }

    // the epilogue warps' C stores have read their staging boxes
    if (warp >= 2 && lane == 0) ptx::bulk_wait_group_read0();
    // no CTA leaves while its partner may still signal its barriers, read its
    // shared memory or write its tensor memory
    __syncwarp();
    __syncthreads();
    ptx::cluster_arrive_release();
    ptx::cluster_wait();
    __syncwarp();
    if (warp == 1) {
        ptx::tc_fence_after();
        tmem_dealloc_pair(tmem, 512);
    }
}

// W4A16 weights dequantised to bf16: W[n,k] = (q[n,k] - z[n,k/g]) * s[n,k/g],
// the product exact in fp32 and rounded once to bf16 (nearest even).  One
// thread per 16 bytes of packed words (32 weights of one group, since g is a
// multiple of 32): a 16-byte streaming load, four 16-byte stores.
__global__ void __launch_bounds__(256) k_w4_dequant(const uint4 *__restrict__ bq, const uint16_t *__restrict__ scales,
                                                    const uint8_t *__restrict__ zeros, uint4 *__restrict__ w,
                                                    int64_t chunks, int cpr, int G, int lg_group)
{
    ptx::pdl_wait();   // the previous kernel may still read the buffer
    ptx::pdl_launch_dependents();
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < chunks; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t n = i / cpr;
        const int k0 = (int)(i - n * cpr) * 32;
        const int grp = k0 >> lg_group;
        const float s = bf16lo(__ldg(scales + n * G + grp));
        const float z = (float)__ldg(zeros + n * G + grp);
        const uint4 q = ld_stream_v4(bq + i);
        const uint32_t words[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {   // word j: weights k0 + 8j .. k0 + 8j + 7
            uint4 o;
            uint32_t *op = reinterpret_cast<uint32_t *>(&o);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float lo = ((float)((words[j] >> (8 * e)) & 0xFu) - z) * s;
                const float hi = ((float)((words[j] >> (8 * e + 4)) & 0xFu) - z) * s;
                op[e] = pack_bf16x2_rn(lo, hi);
            }
            w[i * 4 + j] = o;
        }
    }
}

}  // namespace

// W4A16 at prefill sizes: dequantise the weights once into the workspace
// (bf16 [N, K], after the stream-K partials), then the pair GEMM on them.
cudaError_t launch_w4_pair(const GemmArgs &a, const Plan &p, const LaunchCtx &c)
{
    if (!c.act_copy) return cudaErrorInvalidValue;
    uint16_t *W = (uint16_t *)c.act_copy;
    const int64_t chunks = a.N * (a.K / 32);
    int64_t grid = (chunks + 255) / 256;
    if (grid > (int64_t)c.sm_count * 16) grid = (int64_t)c.sm_count * 16;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = c.stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, k_w4_dequant, (const uint4 *)a.B, (const uint16_t *)a.scales,
                                       (const uint8_t *)a.zeros, (uint4 *)W, chunks, (int)(a.K / 32),
                                       (int)(a.K / a.group), a.group == 32 ? 5 : a.group == 64 ? 6 : 7);
    if (e != cudaSuccess) return e;
    GemmArgs b = a;
    b.B = W;
    b.ldb = a.K;
    b.lda = a.K;
    b.ldc = a.N;
    return launch_umma_pair(b, p, c);
}

// Pair plan (tiles of 256 x 256, the pairs are the schedule's CTAs, at most
// one pair per two SMs):
//   - a last wave holding a quarter to half of the pairs, on a long K: the
//     full waves run whole tiles and each leftover tile is split along K among
//     S = 2 or 3 pairs (stream-K over those), so the last wave ends after 1/S
//     of a tile.  The split pays only when the time it saves, (1 - 1/S) of a
//     tile's k-blocks, exceeds the cost of the fixup (partials written and
//     summed, about 15 us, as long as 48 k-blocks at the MMA rate), measured
//     on GB300: 4096 x 4096 x 12288 +5-10%, 768 x 8192 x 8192 +5-20%, while
//     1024 x 6144 x 4096, 4096 x 4096 x 4096 and 512 x 14336 x 4096 (K = 4096,
//     64 k-blocks) ran 5-10% slower split than as whole tiles;
//   - tiles for at least half the pairs: whole tiles round-robin;
//   - fewer: stream-K over every pair.
// Sets mode, grid (CTAs, two per pair), whole, sk_grid (pairs) and split.
void plan_pair(int64_t M, int64_t N, int64_t K, int sm_count, Plan *p)
{
    constexpr int64_t kFixupKBlocks = 48;
    const int64_t tiles = ((M + 255) / 256) * ((N + BN - 1) / BN);
    const int64_t nk = (K + BK - 1) / BK;
    const int64_t pairs = std::max(1, sm_count / 2);
    const int64_t rem = tiles % pairs;
    const int64_t S = rem ? std::min<int64_t>({3, pairs / rem, nk}) : 1;
    p->whole = 0;
    p->sk_grid = 0;
    p->group_r = 0;
    if (tiles > pairs && rem * 4 > pairs && rem * 2 <= pairs && S >= 2 && (S - 1) * nk > kFixupKBlocks * S) {
        p->mode = 1;
        p->grid = (int)(2 * pairs);
        p->whole = (int)(tiles - rem);
        p->sk_grid = (int)(rem * S);
        p->split = (int)S;
    } else if (2 * tiles >= pairs || tiles * nk < 2 * pairs) {
        p->mode = 0;
        p->grid = (int)(2 * std::min(tiles, pairs));
        p->split = 1;
    } else {
        // token tiles in lockstep (as in the single-CTA planner): tile-rows in
        // order and a multiple of them sharing the units
        const int64_t tiles_r = (M + 255) / 256;
        const bool lock = tiles_r > 1 && pairs >= 2 * tiles_r;
        const int64_t sk = lock ? pairs / tiles_r * tiles_r : pairs;
        p->mode = 1;
        p->grid = (int)(2 * sk);
        p->sk_grid = (int)sk;
        p->group_r = lock ? 1 : 0;
        const int64_t per_pair = tiles * nk / sk;   // >= 2
        p->split = (int)std::min<int64_t>(sk, (nk + per_pair - 1) / per_pair + 1);
    }
}

cudaError_t launch_umma_pair(const GemmArgs &a, const Plan &p, const LaunchCtx &c)
{
    // with the SiLU-mul epilogue B holds 2N rows (gate, then up) and a tile
    // covers 128 output columns through the (gate, up) row-pair view
    const bool pairs = a.epi == GEMM_EPI_SILU_MUL;
    const bool grp = a.gends != nullptr;   // grouped: B stacks the experts' weights [groups * N, K]
    if (grp && (pairs || a.groups < 1 || a.groups > kPairMaxExperts || p.mode != 0)) return cudaErrorInvalidValue;
    CUtensorMap ma, mb, mc;
    if (!make_map_bf16(&ma, a.A, a.M, a.K, a.lda, BMC) ||
        !(pairs ? make_map_pairs(&mb, a.B, a.N, a.K, a.ldb, BNC / 2)
                : make_map_bf16(&mb, a.B, grp ? a.groups * a.N : a.N, a.K, a.ldb, BNC)) ||
        !(pairs ? make_map_c16(&mc, a.C, a.M, a.N, a.ldc) : make_map_c32(&mc, a.C, a.M, a.N, a.ldc)))
        return cudaErrorInvalidValue;
    if (epi_has_bias(a.epi) && !a.bias) return cudaErrorInvalidValue;
    Sched s{};
    s.mode = p.mode;
    s.tiles_r = (int)((a.M + 255) / 256);
    s.tiles_q = (int)((a.N + (pairs ? BN / 2 : BN) - 1) / (pairs ? BN / 2 : BN));
    // grouped: at most one partial m-tile per expert beyond the M / 256 full
    // ones (the tiles are found on the device)
    s.tiles = (grp ? s.tiles_r + (int)a.groups : s.tiles_r) * s.tiles_q;
    s.nk = (int)((a.K + BK - 1) / BK);
    s.grid = p.grid / 2;   // the schedule's CTAs are the pairs
    s.group_r = p.mode == 1 && p.group_r > 0 ? p.group_r : std::min(s.tiles_r, 8);
    s.whole = s.mode == 1 ? p.whole : 0;
    s.sk_grid = s.mode == 1 ? std::min(p.sk_grid, s.grid) : 0;
    s.units = (long long)(s.tiles - s.whole) * s.nk;
    s.stall = g_debug_stall;
    s.epi = a.epi;
    s.pairs = pairs ? 1 : 0;
    s.bias = (const uint16_t *)a.bias;
    s.gends = a.gends;
    s.groups = (int)a.groups;
    s.gN = (int)a.N;
    if (s.mode == 1 && (!c.workspace || !c.counters)) return cudaErrorInvalidValue;
    auto kern = pairs ? k_umma_pair<true, false> : grp ? k_umma_pair<false, true> : k_umma_pair<false, false>;
    const int ki = pairs ? 1 : grp ? 2 : 0;
    static std::once_flag once[3][64];
    static cudaError_t attr_err[3][64];
    int dev = 0;
    cudaGetDevice(&dev);
    std::call_once(once[ki][dev & 63], [&] {
        attr_err[ki][dev & 63] = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    });
    if (attr_err[ki][dev & 63] != cudaSuccess) return attr_err[ki][dev & 63];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.grid, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = SMEM;
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
    return cudaLaunchKernelEx(&cfg, kern, ma, mb, mc, (uint16_t *)a.C, a.ldc, (int)a.M, (int)a.N, s, c.workspace,
                              c.counters, c.d_error);
}

}  // namespace dbw
