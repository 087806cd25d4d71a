// mxgemm.cu -- the block-scaled (microscaling, "MX") GEMM on the 5th-generation
// tensor core:  C[m,n] = sum_k (a[m,k] 2^(sa[m,k/32]-127)) (b[n,k] 2^(sb[n,k/32]-127)).
//
// FlyDSL-in-PyTorch blog, section "MXFP": operands FP8 E4M3 or packed FP4
// E2M1, one E8M0 scale per 32 values along the reduction axis, fp32
// accumulation, bf16 output, K a multiple of 128, unit stride along K for A
// and B.  The scales are applied by the MMA itself
// (tcgen05.mma ... .block_scale): E4M3 x E4M3 with kind::mxf8f6f4 (K = 32 per
// MMA, one scale per row per MMA), packed E2M1 x E2M1 with kind::mxf4 (K = 64
// per MMA, two scales per row per MMA).
//
// Roles (192 threads, one CTA per SM, persistent over tiles of 128 rows of A
// x BN rows of B):
//   warp 0      producer: per stage one 128-byte-wide K slice of the A and B
//               tiles (TMA, 128-byte swizzle: 128 fp8 or 256 fp4 values per
//               row) and the stage's scale-factor chunks (bulk copies)
//   warp 1      MMA issuer: copies the stage's scale factors from shared to
//               tensor memory (tcgen05.cp), then four block-scaled MMAs
//   warps 2-5   epilogue: tensor memory -> registers -> bf16 stores (or the
//               stream-K partial and its deterministic fixup)
//
// Scale factors.  The MMA reads them from tensor memory in the layout that
// tcgen05.cp ... 32x128b.warpx4 produces from a 512-byte chunk of 128 rows x
// 4 consecutive 32-value blocks: byte (r % 32) * 16 + (r / 32) * 4 + j for row
// r and block j (the copy replicates the 32 x 16-byte chunk into all four lane
// quarters; column q of a lane holds rows 32 q + lane).  A pre-pass kernel
// rearranges the caller's row-major [rows, K/32] scales into such chunks,
// ordered [k chunk][row block], so that the two row blocks of a 256-row B
// tile are one contiguous 1 KB copy.  Within a chunk the MMA's scale-factor
// ID picks the block: E4M3 MMA j (K = 32) uses block j; E2M1 MMA j (K = 64)
// uses blocks 2(j % 2) and 2(j % 2) + 1 of chunk j / 2.
//
// Tensor memory: the accumulator(s) at column 0 (two of BN columns when BN =
// 128, one when BN = 256), then a ring of eight 32-column scale-factor slots
// from column 256 (A's chunks at +0, B's at +8 in each slot).  The copies and
// MMAs of one thread execute in issue order, so a stage's MMAs see its
// scale factors; a slot is rewritten eight stages later.
//
// Every wait is bounded (waits.cuh), as in the other TMA-fed kernels.
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

constexpr int BM = kTileRows;
constexpr int kStageBytesK = 128;   // bytes of each A / B row per stage
constexpr int kSfSlots = 8;
constexpr uint32_t kSfCol = 256;
constexpr int kEpiThreads = 128;

template <int FMT>   // 0: E4M3 x E4M3, 1: packed E2M1 x E2M1
struct MxKind {
    static constexpr int KSTAGE = FMT == 0 ? 128 : 256;        // k per stage (128 bytes per row)
    static constexpr int CHUNKS = KSTAGE / 128;                // 4-block scale chunks per stage
    static constexpr uint32_t ATYPE = FMT == 0 ? 0u : 1u;      // E4M3 (mxf8f6f4) / E2M1 (mxf4)
};

// Instruction descriptor of a block-scaled MMA: scale-factor IDs of B (bits
// 4-5) and A (bits 29-30), A and B types (bits 7-9, 10-12), both K-major
// (bits 15, 16 = 0), N >> 3 (bits 17-22), scale type E8M0 (bit 23 = 1),
// M >> 4 (bits 24-28).
__host__ __device__ constexpr uint32_t idesc_mx(uint32_t atype, uint32_t btype, int m, int n, uint32_t sfa_id,
                                                 uint32_t sfb_id)
{
    return (sfb_id << 4) | (atype << 7) | (btype << 10) | ((uint32_t)(n >> 3) << 17) | (1u << 23) |
           ((uint32_t)(m >> 4) << 24) | (sfa_id << 29);
}

template <int FMT>
__device__ __forceinline__ void mma_mx_warp(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t sfa,
                                            uint32_t sfb, uint32_t accumulate)
{
    if constexpr (FMT == 0) {
        asm volatile(
            "{\n\t.reg .pred p, e;\n\t"
            "elect.sync _|e, 0xffffffff;\n\t"
            "setp.ne.b32 p, %6, 0;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::
                "r"(d),
            "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
            : "memory");
    } else {
        asm volatile(
            "{\n\t.reg .pred p, e;\n\t"
            "elect.sync _|e, 0xffffffff;\n\t"
            "setp.ne.b32 p, %6, 0;\n\t"
            "@e tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::
                "r"(d),
            "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
            : "memory");
    }
}

// 32 rows x 16 bytes of shared memory -> 4 tensor-memory columns, replicated
// into all four lane quarters, from one elected lane of a converged warp.
// The shared-memory descriptor: start >> 4, no swizzle, core matrices of 8
// rows x 16 bytes one after another (stride 128 bytes), version 1.
__device__ __forceinline__ void sf_copy_warp(uint32_t taddr, uint32_t saddr)
{
    const uint64_t desc = (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(128 >> 4) << 32) |
                          ((uint64_t)1 << 46);
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;\n\t}" ::"r"(taddr),
        "l"(desc)
        : "memory");
}

// Shared memory: a ring of STAGES data stages (A tile, then B tile; 1024-byte
// aligned for the swizzle), then a ring of the stages' scale chunks (A's,
// then B's).
template <int BN, int FMT>
struct MxLayout {
    static constexpr int STAGES = 4;
    static constexpr int A_BYTES = BM * kStageBytesK;         // 16 KB
    static constexpr int B_BYTES = BN * kStageBytesK;         // 16 or 32 KB
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;     // multiple of 1024
    static constexpr int SFA_BYTES = MxKind<FMT>::CHUNKS * 512;
    static constexpr int SFB_BYTES = MxKind<FMT>::CHUNKS * (BN / 128) * 512;
    static constexpr int SF_OFF = STAGES * STAGE_BYTES;
    static constexpr int SF_STAGE = SFA_BYTES + SFB_BYTES;
    static constexpr int BAR_OFF = SF_OFF + STAGES * SF_STAGE;
    static constexpr int NACC = BN == 128 ? 2 : 1;
    static constexpr int NBARS = 2 * STAGES + 2 * NACC + 2;
    static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;
    static constexpr int SMEM = MISC_OFF + 16 + 1024;
    static_assert(STAGE_BYTES % 1024 == 0, "stages keep the 1024-byte swizzle alignment");
    static_assert(NACC * BN <= (int)kSfCol, "tensor-memory map");
};

struct MxArgs {
    const uint8_t *sfa;   // A's scale chunks [K/128 (padded)][row blocks of A][512]
    const uint8_t *sfb;   // B's scale chunks [K/128 (padded)][row blocks of B][512]
    int rba, rbb;         // row blocks (of 128) in each chunk row
};

template <int BN, int FMT>
__global__ void __launch_bounds__(192, 1)
k_mx(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, uint16_t *__restrict__ C, int R,
     int Q, int64_t ldc, const __grid_constant__ Sched sched, const MxArgs mx, float *__restrict__ ws,
     int *__restrict__ counters, int *__restrict__ d_error)
{
    using L = MxLayout<BN, FMT>;
    using KD = MxKind<FMT>;
    constexpr int STAGES = L::STAGES, NACC = L::NACC;
    extern __shared__ uint8_t mx_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(mx_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = ptx::smem_addr(smem);
    const uint32_t bar0 = sbase + (uint32_t)L::BAR_OFF;
    auto FULL = [&](int s) { return bar0 + 8u * s; };
    auto EMPTY = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto TFULL = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
    auto TEMPTY = [&](int a) { return bar0 + 8u * (2 * STAGES + NACC + a); };
    const uint32_t DONE = bar0 + 8u * (2 * STAGES + 2 * NACC);
    const uint32_t FIXB = bar0 + 8u * (2 * STAGES + 2 * NACC + 1);   // epilogue warps' barrier
    uint32_t *misc = reinterpret_cast<uint32_t *>(smem + L::MISC_OFF);   // [0] tmem, [1] abort, [2] last flag
    volatile uint32_t *abort_flag = misc + 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(FULL(s), 1);
            ptx::mbar_init(EMPTY(s), 1);
        }
        for (int a = 0; a < NACC; ++a) {
            ptx::mbar_init(TFULL(a), 1);
            ptx::mbar_init(TEMPTY(a), kEpiThreads / 32);
        }
        ptx::mbar_init(DONE, 1);
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
        ptx::prefetch_tmap(&tmA);
        ptx::prefetch_tmap(&tmB);
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = misc[0];
    ptx::pdl_launch_dependents();

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            ptx::pdl_wait();   // the scale chunks come from the pre-pass
            const uint64_t pol_a = ptx::policy_evict_last();
            const uint64_t pol_b = sched.tiles_r == 1 ? ptx::policy_evict_first() : ptx::policy_evict_last();
            long long gs = 0, issued = 0;
            SegIter it(sched, blockIdx.x, sched.tiles);
            Segment seg;
            bool ok = true;
            while (ok && it.next(sched, seg)) {
                int tr, tq;
                tile_coords(sched, seg.tile, tr, tq);
                for (int kb = seg.kb0; kb < seg.kb1; ++kb, ++gs) {
                    const int s = (int)(gs % STAGES);
                    if (!wait_bar(EMPTY(s), (uint32_t)(((gs / STAGES) & 1) ^ 1), abort_flag, d_error)) {
                        ok = false;
                        break;
                    }
                    if (sched.stall) continue;
                    const uint32_t st = sbase + (uint32_t)(s * L::STAGE_BYTES);
                    const uint32_t sf = sbase + (uint32_t)(L::SF_OFF + s * L::SF_STAGE);
                    ptx::mbar_arrive_expect_tx(FULL(s), (uint32_t)(L::STAGE_BYTES + L::SF_STAGE));
                    ptx::tma_load_2d(st, &tmA, FULL(s), kb * kStageBytesK, tr * BM, pol_a);
                    ptx::tma_load_2d(st + L::A_BYTES, &tmB, FULL(s), kb * kStageBytesK, tq * BN, pol_b);
#pragma unroll
                    for (int c = 0; c < KD::CHUNKS; ++c) {
                        const int kc = kb * KD::CHUNKS + c;
                        bulk_load(sf + c * 512, mx.sfa + ((int64_t)kc * mx.rba + tr) * 512, 512, FULL(s));
                        bulk_load(sf + L::SFA_BYTES + c * (BN / 128) * 512,
                                  mx.sfb + ((int64_t)kc * mx.rbb + tq * (BN / 128)) * 512, (BN / 128) * 512, FULL(s));
                    }
                    ++issued;
                }
            }
            if (!ok) {
                for (int s = 0; s < STAGES; ++s) {
                    if (issued <= s) continue;
                    const long long last = issued - 1 - ((issued - 1 - s) % STAGES);
                    wait_bar_drain(FULL(s), (uint32_t)((last / STAGES) & 1));
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        long long gs = 0;
        int acc = 0;
        uint32_t acc_phase = 0;
        SegIter it(sched, blockIdx.x, sched.tiles);
        Segment seg;
        bool ok = true;
        while (ok && it.next(sched, seg)) {
            if (!wait_bar_warp(TEMPTY(acc), acc_phase ^ 1u, abort_flag, d_error)) break;
            ptx::tc_fence_after();
            const uint32_t d = tmem + (uint32_t)(acc * BN);
            for (int kb = seg.kb0; kb < seg.kb1; ++kb, ++gs) {
                const int s = (int)(gs % STAGES);
                if (!wait_bar_warp(FULL(s), (uint32_t)((gs / STAGES) & 1), abort_flag, d_error)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t st = sbase + (uint32_t)(s * L::STAGE_BYTES);
                const uint32_t sfs = sbase + (uint32_t)(L::SF_OFF + s * L::SF_STAGE);
                const uint32_t slot = tmem + kSfCol + (uint32_t)((gs % kSfSlots) * 32);
#pragma unroll
                for (int c = 0; c < KD::CHUNKS; ++c) {
                    sf_copy_warp(slot + (uint32_t)(4 * c), sfs + (uint32_t)(c * 512));
#pragma unroll
                    for (int h = 0; h < BN / 128; ++h)
                        sf_copy_warp(slot + 8u + (uint32_t)(4 * ((BN / 128) * c + h)),
                                     sfs + L::SFA_BYTES + (uint32_t)(((BN / 128) * c + h) * 512));
                }
                const uint64_t ad = ptx::sdesc_kmajor_sw128(st), bd = ptx::sdesc_kmajor_sw128(st + L::A_BYTES);
#pragma unroll
                for (int j = 0; j < 4; ++j) {   // 32 bytes of each row per MMA
                    const int c = FMT == 0 ? 0 : j >> 1;                       // chunk of this MMA's blocks
                    const uint32_t sid = FMT == 0 ? (uint32_t)j : (uint32_t)(2 * (j & 1));
                    const uint32_t idesc = idesc_mx(KD::ATYPE, KD::ATYPE, BM, BN, sid, sid);
                    mma_mx_warp<FMT>(d, ad + 2u * j, bd + 2u * j, idesc, slot + (uint32_t)(4 * c),
                                     slot + 8u + (uint32_t)(4 * (BN / 128) * c), (kb > seg.kb0 || j > 0) ? 1u : 0u);
                }
                ptx::mma_commit_warp(EMPTY(s));
            }
            if (!ok) break;
            ptx::mma_commit_warp(TFULL(acc));
            if (++acc == NACC) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        ptx::mma_commit_warp(DONE);
        wait_bar_drain(DONE, 0);
    } else {
        // ------------------------------------------------------------ epilogue (warps 2-5)
        const int q4 = warp & 3;
        const int row = q4 * 32 + lane;
        const int etid = threadIdx.x - 64;
        ptx::pdl_wait();
        int acc = 0;
        uint32_t acc_phase = 0, fphase = 0;
        SegIter it(sched, blockIdx.x, sched.tiles);
        Segment seg;
        while (it.next(sched, seg)) {
            if (!wait_bar_warp(TFULL(acc), acc_phase, abort_flag, d_error)) break;
            ptx::tc_fence_after();
            int tr, tq;
            tile_coords(sched, seg.tile, tr, tq);
            const int r = tr * BM + row, qb = tq * BN;
            const uint32_t taddr = tmem + ((uint32_t)(q4 * 32) << 16) + (uint32_t)(acc * BN);
            const bool whole = seg.kb0 == 0 && seg.kb1 == sched.nk;
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
                    store_chunk<false>(C, ldc, R, Q, r, qb + c, f);
                } else {
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        __stcg(part + (c / 4 + u) * BM + row, make_float4(f[4 * u], f[4 * u + 1], f[4 * u + 2], f[4 * u + 3]));
                }
            }
            ptx::tc_fence_before();
            arrive_warp(TEMPTY(acc));
            if (++acc == NACC) {
                acc = 0;
                acc_phase ^= 1u;
            }
            if (whole) continue;
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
            streamk_fixup<BN, 16>(sched, ws, t, row, [&](int c0, const float(&f)[16]) {
                store_chunk<false>(C, ldc, R, Q, r, qb + c0, f);
            });
        }
    }

    __syncwarp();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
}

// Row-major E8M0 scales [rows, K/32] -> chunks [kc][row block][512 bytes]:
// byte (r % 32) * 16 + (r / 32) * 4 + j of chunk (kc, rb) is the scale of row
// 128 rb + r, block 4 kc + j (zero past the last row or the last block).  One
// thread per (chunk, row): four scale bytes, one 4-byte store.
__global__ void __launch_bounds__(256) k_mx_sf_prep(const uint8_t *__restrict__ sa, uint8_t *__restrict__ ca, int rows_a,
                                                    int rba, const uint8_t *__restrict__ sb, uint8_t *__restrict__ cb,
                                                    int rows_b, int rbb, int kcs, int kcp)
{
    ptx::pdl_wait();   // the previous kernel may still read the chunks
    ptx::pdl_launch_dependents();
    const int64_t na = (int64_t)kcp * rba * 128, nb = (int64_t)kcp * rbb * 128;
    const int nblk = kcs * 4;   // 32-value blocks per row
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < na + nb; i += (int64_t)gridDim.x * blockDim.x) {
        const bool isa = i < na;
        const int64_t li = isa ? i : i - na;
        const int rb_n = isa ? rba : rbb;
        const int r = (int)(li % 128);
        const int64_t cr = li / 128;           // chunk index kc * rb_n + rb
        const int rb = (int)(cr % rb_n), kc = (int)(cr / rb_n);
        const int row = rb * 128 + r;
        const int rows = isa ? rows_a : rows_b;
        const uint8_t *src = isa ? sa : sb;
        uint32_t v = 0;
        if (row < rows && kc < kcs) v = __ldg(reinterpret_cast<const uint32_t *>(src + (int64_t)row * nblk) + kc);
        uint8_t *dst = (isa ? ca : cb) + cr * 512 + (r % 32) * 16 + (r / 32) * 4;
        *reinterpret_cast<uint32_t *>(dst) = v;
    }
}

template <int BN, int FMT>
cudaError_t launch_mx_t(const CUtensorMap &ma, const CUtensorMap &mb, uint16_t *C, int R, int Q, int64_t ldc,
                        const Sched &s, const MxArgs &mx, const LaunchCtx &c)
{
    using L = MxLayout<BN, FMT>;
    auto kern = k_mx<BN, FMT>;
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
    cfg.blockDim = dim3(192, 1, 1);
    cfg.dynamicSmemBytes = L::SMEM;
    cfg.stream = c.stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, ma, mb, C, R, Q, ldc, s, mx, c.workspace, c.counters, c.d_error);
}

}  // namespace

int mx_stage_k(int fmt) { return fmt == 0 ? MxKind<0>::KSTAGE : MxKind<1>::KSTAGE; }

int64_t mx_sf_workspace_bytes(int64_t M, int64_t N, int64_t K, int fmt, int bn)
{
    const int64_t kcp = (K + mx_stage_k(fmt) - 1) / mx_stage_k(fmt) * (mx_stage_k(fmt) / 128);
    const int64_t rba = (M + 127) / 128, rbb = (N + bn - 1) / bn * (bn / 128);
    return kcp * (rba + rbb) * 512;
}

cudaError_t launch_mx(const GemmArgs &a, const Plan &p, const LaunchCtx &c, int fmt)
{
    if (!c.act_copy || (p.mode == 1 && (!c.workspace || !c.counters))) return cudaErrorInvalidValue;
    const int bn = p.bn;
    const int64_t kst = mx_stage_k(fmt);
    const int kcs = (int)(a.K / 128);
    const int kcp = (int)((a.K + kst - 1) / kst * (kst / 128));
    const int rba = (int)((a.M + 127) / 128), rbb = (int)((a.N + bn - 1) / bn * (bn / 128));
    uint8_t *ca = (uint8_t *)c.act_copy;
    uint8_t *cb = ca + (int64_t)kcp * rba * 512;
    {
        const int64_t items = (int64_t)kcp * (rba + rbb) * 128;
        int64_t grid = (items + 255) / 256;
        if (grid > (int64_t)c.sm_count * 8) grid = (int64_t)c.sm_count * 8;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)grid, 1, 1);
        cfg.blockDim = dim3(256, 1, 1);
        cfg.stream = c.stream;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        at[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        cudaError_t e = cudaLaunchKernelEx(&cfg, k_mx_sf_prep, (const uint8_t *)a.sfa, ca, (int)a.M, rba,
                                           (const uint8_t *)a.sfb, cb, (int)a.N, rbb, kcs, kcp);
        if (e != cudaSuccess) return e;
    }
    const int64_t width_bytes = fmt == 0 ? a.K : a.K / 2;
    CUtensorMap ma, mb;
    if (!make_map_u8(&ma, a.A, a.M, width_bytes, BM) || !make_map_u8(&mb, a.B, a.N, width_bytes, bn))
        return cudaErrorInvalidValue;
    Sched s{};
    s.mode = p.mode;
    s.tiles_r = (int)((a.M + BM - 1) / BM);
    s.tiles_q = (int)((a.N + bn - 1) / bn);
    s.tiles = s.tiles_r * s.tiles_q;
    s.nk = (int)((a.K + kst - 1) / kst);
    s.grid = p.grid;
    s.group_r = p.group_r > 0 ? p.group_r : s.tiles_r;
    s.whole = 0;
    s.sk_grid = p.grid;
    s.units = (long long)s.tiles * s.nk;
    s.stall = g_debug_stall;
    s.split = p.split;
    MxArgs mx{ca, cb, rba, rbb};
    uint16_t *C = (uint16_t *)a.C;
    const int R = (int)a.M, Q = (int)a.N;
    if (fmt == 0)
        return bn == 128 ? launch_mx_t<128, 0>(ma, mb, C, R, Q, a.ldc, s, mx, c)
                         : launch_mx_t<256, 0>(ma, mb, C, R, Q, a.ldc, s, mx, c);
    return bn == 128 ? launch_mx_t<128, 1>(ma, mb, C, R, Q, a.ldc, s, mx, c)
                     : launch_mx_t<256, 1>(ma, mb, C, R, Q, a.ldc, s, mx, c);
}

}  // namespace dbw
