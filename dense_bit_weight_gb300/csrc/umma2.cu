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
// Roles (192 threads per CTA, one CTA per SM, persistent over pair tiles):
//   warp 0      producer, in both CTAs: per stage the CTA's 128 rows of A and
//               its 128 rows of B (TMA, 128-byte swizzle), both copies
//               signalling the LEADER's full barrier (the .cta_group::2 form);
//               the leader's producer announces the bytes of both CTAs
//   warp 1      allocates the pair's tensor memory (both CTAs); in the leader
//               issues four MMAs (K = 16) per stage and commits the stage's
//               release and the accumulator's completion to the barriers of
//               both CTAs (multicast)
//   warps 2-5   epilogue, in both CTAs: the CTA's 128 accumulator rows ->
//               bf16 -> C; each warp then releases the accumulator on the
//               leader's barrier (eight arrivals: four local, four remote)
// Two accumulators of 256 columns let the epilogue of one tile overlap the
// MMAs of the next.  Every wait is bounded (waits.cuh); a cluster barrier
// before exit keeps either CTA from leaving while its partner may still
// signal its barriers or read its shared memory.
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

constexpr int BMC = kTileRows;      // A rows per CTA (256 per pair)
constexpr int BN = 256;             // B rows per pair tile (128 per CTA)
constexpr int BNC = BN / 2;
constexpr int BK = 64;
constexpr int STAGES = 6;
constexpr int A_BYTES = BMC * BK * 2;    // 16 KB
constexpr int B_BYTES = BNC * BK * 2;    // 16 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int BAR_OFF = STAGES * STAGE_BYTES;
constexpr int NBARS = 2 * STAGES + 4 + 1;
constexpr int MISC_OFF = BAR_OFF + NBARS * 8;
constexpr int SMEM = MISC_OFF + 16 + 1024;
constexpr int kEpiThreads = 128;

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

__global__ void __launch_bounds__(192, 1)
k_umma_pair(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, uint16_t *__restrict__ C,
            int M, int N, int64_t ldc, const __grid_constant__ Sched sched, int *__restrict__ d_error)
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
    uint32_t *misc = reinterpret_cast<uint32_t *>(smem + MISC_OFF);   // [0] tmem, [1] abort
    volatile uint32_t *abort_flag = misc + 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = ptx::cluster_ctarank();
    const bool leader = rank == 0;
    const int pair = (int)(blockIdx.x >> 1), npairs = (int)(gridDim.x >> 1);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(FULL(s), 1);    // the leader's producer; both CTAs' copies count their bytes
            ptx::mbar_init(EMPTY(s), 1);   // the leader's multicast commit
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(TFULL(a), 1);
            ptx::mbar_init(TEMPTY(a), 2 * kEpiThreads / 32);   // (used in the leader) both CTAs' epilogue warps
        }
        ptx::mbar_init(DONE, 1);
        misc[1] = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(ptx::smem_addr(misc), 512);
        tmem_relinquish_pair();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tmA);
        ptx::prefetch_tmap(&tmB);
    }
    ptx::tc_fence_before();
    // both CTAs' barriers are initialised before any copy or commit signals them
    ptx::cluster_arrive_release();
    ptx::cluster_wait();
    __syncwarp();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = misc[0];
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
            for (int t = pair; ok && t < sched.tiles; t += npairs) {
                int tm, tn;
                tile_coords(sched, t, tm, tn);
                for (int kb = 0; kb < sched.nk; ++kb) {
                    if (!wait_bar(EMPTY(stage), phase ^ 1u, abort_flag, d_error)) {
                        ok = false;
                        break;
                    }
                    if (!sched.stall) {
                        const uint32_t full = ptx::map_cluster(FULL(stage), 0u);   // the leader's barrier
                        if (leader) ptx::mbar_arrive_expect_tx(FULL(stage), 2u * STAGE_BYTES);
                        const uint32_t st = sbase + (uint32_t)(stage * STAGE_BYTES);
                        tma_load_pair(st, &tmA, full, kb * BK, tm * (2 * BMC) + (int)rank * BMC, pol_a);
                        tma_load_pair(st + A_BYTES, &tmB, full, kb * BK, tn * BN + (int)rank * BNC, pol_b);
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
            for (int t = pair; ok && t < sched.tiles; t += npairs) {
                if (!wait_bar_warp(TEMPTY(acc), acc_phase ^ 1u, abort_flag, d_error)) break;
                ptx::tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(acc * BN);
                for (int kb = 0; kb < sched.nk; ++kb) {
                    if (!wait_bar_warp(FULL(stage), phase, abort_flag, d_error)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t st = sbase + (uint32_t)(stage * STAGE_BYTES);
                    const uint64_t ad = ptx::sdesc_kmajor_sw128(st), bd = ptx::sdesc_kmajor_sw128(st + A_BYTES);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k)
                        mma_pair_warp(d, ad + 2u * k, bd + 2u * k, IDESC, (kb > 0 || k > 0) ? 1u : 0u);
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
        const int q4 = warp & 3;
        const int row = q4 * 32 + lane;
        ptx::pdl_wait();
        const uint32_t temp_leader0 = ptx::map_cluster(TEMPTY(0), 0u);
        const uint32_t temp_leader1 = ptx::map_cluster(TEMPTY(1), 0u);
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int t = pair; t < sched.tiles; t += npairs) {
            if (!wait_bar_warp(TFULL(acc), acc_phase, abort_flag, d_error)) break;
            ptx::tc_fence_after();
            int tm, tn;
            tile_coords(sched, t, tm, tn);
            const int r = tm * (2 * BMC) + (int)rank * BMC + row;
            const uint32_t taddr = tmem + ((uint32_t)(q4 * 32) << 16) + (uint32_t)(acc * BN);
#pragma unroll 1
            for (int c = 0; c < BN; c += 16) {
                uint32_t v[16];
                __syncwarp();
                ptx::tmem_ld16(taddr + (uint32_t)c, v);
                ptx::tmem_wait_ld();
                float f[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) f[j] = __uint_as_float(v[j]);
                store_chunk<false>(C, ldc, M, N, r, tn * BN + c, f);
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) arrive_remote(acc == 0 ? temp_leader0 : temp_leader1);
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
    }

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
// (bf16 [N, K]), then the pair GEMM on them.
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

// Pair tiles for the prefill shapes: 256 x 256 tiles in a grouped raster,
// whole tiles round-robin over the pairs (two CTAs per pair, at most one pair
// per two SMs).
int umma_pair_grid(int64_t M, int64_t N, int sm_count)
{
    const int64_t tiles = ((M + 255) / 256) * ((N + BN - 1) / BN);
    return (int)std::min<int64_t>(tiles, sm_count / 2) * 2;
}

cudaError_t launch_umma_pair(const GemmArgs &a, const Plan &p, const LaunchCtx &c)
{
    CUtensorMap ma, mb;
    if (!make_map_bf16(&ma, a.A, a.M, a.K, a.lda, BMC) || !make_map_bf16(&mb, a.B, a.N, a.K, a.ldb, BNC))
        return cudaErrorInvalidValue;
    Sched s{};
    s.mode = 0;
    s.tiles_r = (int)((a.M + 255) / 256);
    s.tiles_q = (int)((a.N + BN - 1) / BN);
    s.tiles = s.tiles_r * s.tiles_q;
    s.nk = (int)((a.K + BK - 1) / BK);
    s.grid = p.grid / 2;   // pairs
    s.group_r = std::min(s.tiles_r, 8);
    s.stall = g_debug_stall;
    static std::once_flag once[64];
    static cudaError_t attr_err[64];
    int dev = 0;
    cudaGetDevice(&dev);
    std::call_once(once[dev & 63], [&] {
        attr_err[dev & 63] = cudaFuncSetAttribute(k_umma_pair, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    });
    if (attr_err[dev & 63] != cudaSuccess) return attr_err[dev & 63];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.grid, 1, 1);
    cfg.blockDim = dim3(192, 1, 1);
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
    return cudaLaunchKernelEx(&cfg, k_umma_pair, ma, mb, (uint16_t *)a.C, (int)a.M, (int)a.N, a.ldc, s, c.d_error);
}

}  // namespace dbw
