// w4frag.cu -- W4A16 for up to 16 tokens: the weights are dequantised into the
// A fragments of warp-level MMAs (mma.sync.m16n8k16, bf16 -> fp32; weight rows
// on the MMA's M side, tokens on its N side) and reach shared memory by TMA.
//
// The contraction is the W4A16 decode GEMM of the hk-dsl PyPI page ("Results",
// W4A16 decode GEMM (AWQ)): w[n,k] = (q[n,k] - z[n,g]) * s[n,g], g = k / group.
// Within one quantisation group the scale and zero are constants, so
//     sum_{k in g} w a = s * D_g + c * S_g,   c = -(128 + z) * s,
//     D_g = sum_{k in g} (128 + q) a,         S_g = sum_{k in g} a.
// 128 + q is exact in bf16 as (0x4300 | q), so the MMA operand needs one mask
// (and for three of the four nibble pairs a shift) per pair of weights; D_g
// accumulates in fp32 in the MMA, and c is exact in fp32 (8-bit s times an
// integer below 144).  The weights are never rounded to bf16.
//
// Work split.  A tile of kW4FragRows weight rows (R blocks of sixteen) is
// shared by P = 1, 2 or 4 warps of one CTA (P chosen so the grid fills the
// device): part p takes the 256-k stages p, p + P, ...  A warp streams its
// stages with TMA -- one 2-D box of 32 words x kW4FragRows rows, 128-byte
// swizzle -- into a ring of its own with one mbarrier per slot and refills a
// slot as soon as it has read it; it stages the next stage's scales and zeros
// as (s, c) pairs in fp32 while it multiplies the current one.  No warp waits
// for another until the P parts of its tile are added, in part order
// (deterministic), through shared memory behind a named barrier of those P
// warps.
//
// Fragment mapping (lane: g = lane / 4, t = lane % 4).  MMA row m of a block
// is weight row 8 (m / 8) + col_row(m % 8), col_row(n) = (n >> 1) | ((n & 1)
// << 2), so the two rows a quarter-warp reads fall in different halves of the
// swizzle pattern and its 16-byte shared loads are conflict-free.  A group is
// 4 WPT words per row (WPT = group / 32); lane t holds words WPT t .. WPT t +
// WPT - 1 of its rows g and g + 8, and its word i feeds k-steps 2i and 2i + 1
// of the group: nibble pairs (0,4) and (1,5) at the fragment's k positions
// (2t, 2t+1) and (2t+8, 2t+9) of k-step 2i, pairs (2,6) and (3,7) in k-step
// 2i + 1.  The activations were copied with every 8-k block in the order
// 0,4,1,5,2,6,3,7 (k_w4_frag_prep), so the B operands of both k-steps of word
// i for token g are one 16-byte load (two register pairs as the MMA takes
// them).  The two k-steps of a word accumulate separately (two independent
// chains per block) and are added at the group's end.
#include <cuda_bf16.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "frag.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "waits.cuh"

namespace dbw {
namespace {

constexpr int kSlots = 3;                      // ring slots (stages in flight) per warp
constexpr int kR = kW4FragRows / 16;           // blocks of sixteen weight rows per CTA
constexpr int kThreads = kW4FragWarps * 32;

// Weight row (within eight) of MMA row n.
__device__ __forceinline__ int col_row(int n) { return (n >> 1) | ((n & 1) << 2); }

__device__ __forceinline__ void mma_first(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%10,%10,%10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}

// Shared-memory layout (from a 1024-byte aligned base: the swizzle pattern
// repeats every 1024 bytes).
template <int NT, int GS>
struct FragLayout {
    static constexpr int SLOT = kW4FragRows * 128;                    // one stage: rows x 128 bytes
    static constexpr int RING = kW4FragWarps * kSlots * SLOT;
    static constexpr int BAR_OFF = RING;                              // [warp][slot] mbarriers
    static constexpr int FLAG_OFF = BAR_OFF + kW4FragWarps * kSlots * 8;
    // per warp, two stages of (s, c): float4 [group][block][g] = (s, c) of the lane's rows g and g + 8
    static constexpr int TAB_OFF = (FLAG_OFF + 16 + 15) / 16 * 16;
    static constexpr int TAB_STAGE = GS * kR * 8 * 16;
    static constexpr int BYTES = TAB_OFF + kW4FragWarps * 2 * TAB_STAGE + 1024;   // + alignment slack
};

// Activations [M, K] -> the copy with every 8-k block in the order
// 0,4,1,5,2,6,3,7, and the group sums S[g, m] (fp32, tokens padded to TP
// with zeros).  One thread per (token < TP, 8-k block); the group/8 threads of
// a group are neighbouring lanes and add their sums by a fixed shuffle tree.
__global__ void __launch_bounds__(256) k_w4_frag_prep(const uint16_t *__restrict__ A, uint16_t *__restrict__ Ap,
                                                      float *__restrict__ S, int M, int TP, int K, int group)
{
    // Every earlier kernel has finished (and no longer reads the workspace)
    // once this returns; only then may the GEMM kernel start reading weights.
    ptx::pdl_wait();
    ptx::pdl_launch_dependents();
    const int KB = K >> 3;   // 8-k blocks per row
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= TP * KB) return;   // TP * KB is a multiple of 32: whole warps leave together
    const int m = i / KB, b = i - m * KB;
    const int bpg = group >> 3;   // blocks per group: 4, 8 or 16 neighbouring lanes
    float sum = 0.f;
    if (m < M) {
        const uint4 a = ld_ro_v4(A + (int64_t)m * K + 8 * b);   // (a0 a1)(a2 a3)(a4 a5)(a6 a7)
        const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) sum += bf16lo(w[j]) + bf16hi(w[j]);
        uint4 o;
        o.x = __byte_perm(a.x, a.z, 0x5410);   // (a0, a4)
        o.y = __byte_perm(a.x, a.z, 0x7632);   // (a1, a5)
        o.z = __byte_perm(a.y, a.w, 0x5410);   // (a2, a6)
        o.w = __byte_perm(a.y, a.w, 0x7632);   // (a3, a7)
        *reinterpret_cast<uint4 *>(Ap + (int64_t)m * K + 8 * b) = o;
    }
    const unsigned seg = __activemask();
    for (int o = 1; o < bpg; o <<= 1) sum += __shfl_xor_sync(seg, sum, o);
    if ((b & (bpg - 1)) == 0) S[(int64_t)(b / bpg) * TP + m] = sum;
}

// NT: token tiles of eight (M <= 8 NT); WPT: group / 32.
template <int NT, int WPT>
__global__ void __launch_bounds__(kThreads, NT == 1 ? 4 : 2)
k_w4_frag(const __grid_constant__ CUtensorMap tmQ, const uint16_t *__restrict__ Ap, const float *__restrict__ S,
          const uint16_t *__restrict__ scales, const uint8_t *__restrict__ zeros, uint16_t *__restrict__ C, int M,
          int N, int K, int P, int *__restrict__ d_error, int stall)
{
    constexpr int GROUP = 32 * WPT;
    constexpr int GS = 8 / WPT;   // groups per 256-k stage
    constexpr int TP = 8 * NT;    // tokens of the MMAs (S is padded to it)
    using L = FragLayout<NT, GS>;
    constexpr int W = kW4FragWarps;
    constexpr int R = kR;
    constexpr int RW = kW4FragRows;
    extern __shared__ uint8_t frag_raw[];
    uint8_t *smem = frag_raw + ((1024u - (ptx::smem_addr(frag_raw) & 1023u)) & 1023u);
    const uint32_t sbase = ptx::smem_addr(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, t = lane & 3;
    const int G = K / GROUP;
    const int nst = (K + 255) >> 8;                  // 256-k stages per tile
    const int tiles = (N + RW - 1) / RW;
    const int wi = blockIdx.x * W + warp;
    const int x = wi / P, part = wi - x * P;         // this warp's tile and part
    const int nu = x < tiles && part < nst ? (nst - 1 - part) / P + 1 : 0;   // its stages: part, part + P, ...
    const uint32_t ring = sbase + (uint32_t)(warp * kSlots * L::SLOT);
    const uint32_t bar0 = sbase + (uint32_t)(L::BAR_OFF + warp * kSlots * 8);
    volatile uint32_t *abort_flag = reinterpret_cast<volatile uint32_t *>(smem + L::FLAG_OFF);
    float *tabw = reinterpret_cast<float *>(smem + L::TAB_OFF + warp * 2 * L::TAB_STAGE);   // this warp's two stages
    const uint64_t policy = ptx::policy_evict_first();
    const int n0 = x * RW;

    // stage j of this warp -> slot j % kSlots (lane 0 only)
    auto issue = [&](int j) {
        const int sl = j % kSlots;
        const uint32_t bar = bar0 + 8u * (uint32_t)sl;
        ptx::mbar_arrive_expect_tx(bar, (uint32_t)L::SLOT);
        ptx::tma_load_2d(ring + (uint32_t)(sl * L::SLOT), &tmQ, bar, (part + P * j) * 32, n0, policy);
    };
    if (threadIdx.x == 0) *abort_flag = 0u;
    if (lane == 0) {
        for (int s = 0; s < kSlots; ++s) ptx::mbar_init(bar0 + 8u * (uint32_t)s, 1);
        ptx::fence_mbar_init();
        ptx::prefetch_tmap(&tmQ);
        // The weights are not written by the preceding kernel (the activation
        // pre-pass), which waited for all earlier work before this grid could
        // start: they may be fetched ahead of the dependency wait.
        if (!stall)
            for (int j = 0; j < kSlots && j < nu; ++j) issue(j);
    }
    // (s, c) of stage st into table slot ts: lane l takes slot row l
    // (block l / 16, MMA row 8 ((l / 8) & 1) + the inverse of col_row(l % 8)) of
    // every group of the stage; sz_load fetches the raw values, sz_store
    // converts and writes them
    const int tab_e = 4 * ((lane >> 4) * 8 + (((lane & 3) << 1) | ((lane >> 2) & 1))) + 2 * ((lane >> 3) & 1);
    const int nrow = n0 + lane;
    auto sz_load = [&](int st, uint32_t (&sr)[GS], uint32_t (&zr)[GS]) {
#pragma unroll
        for (int h = 0; h < GS; ++h) {
            const int gi = st * GS + h;
            const bool v = nrow < N && gi < G;
            sr[h] = v ? (uint32_t)__ldg(scales + (int64_t)nrow * G + gi) : 0u;
            zr[h] = v ? (uint32_t)__ldg(zeros + (int64_t)nrow * G + gi) : 0u;
        }
    };
    auto sz_store = [&](int ts, const uint32_t (&sr)[GS], const uint32_t (&zr)[GS]) {
#pragma unroll
        for (int h = 0; h < GS; ++h) {
            const float sv = __uint_as_float(sr[h] << 16);
            const float cv = -__uint_as_float(0x43000000u | (zr[h] << 16)) * sv;   // -(128 + z) s
            *reinterpret_cast<float2 *>(tabw + ts * (L::TAB_STAGE / 4) + h * (R * 32) + tab_e) = make_float2(sv, cv);
        }
    };
    uint32_t sr[GS], zr[GS];
    if (nu > 0) {
        sz_load(part, sr, zr);
        sz_store(0, sr, zr);
    }
    __syncthreads();   // barriers and the abort flag initialised, first tables written
    ptx::pdl_wait();   // the activation copy and the group sums
    ptx::pdl_launch_dependents();

    float acc[R][NT][4];
#pragma unroll
    for (int b = 0; b < R; ++b)
#pragma unroll
        for (int u = 0; u < NT; ++u)
#pragma unroll
            for (int q = 0; q < 4; ++q) acc[b][u][q] = 0.f;
    const int prow = col_row(g);
    uint32_t woff[GS];   // this lane's words of group h in its row g: logical byte, swizzled by 16-byte piece
#pragma unroll
    for (int h = 0; h < GS; ++h) {
        const int lb = (GROUP / 2) * h + 4 * WPT * t;
        woff[h] = (uint32_t)(prow * 128 + ((((lb >> 4) ^ prow) << 4) | (lb & 15)));
    }
    // B operands of this lane: token 8u + g of the copy, block WPT t of each group;
    // lanes of absent tokens keep zero operands and load nothing
    bool has[NT];
    const uint16_t *ab[NT];
#pragma unroll
    for (int u = 0; u < NT; ++u) {
        has[u] = 8 * u + g < M;
        ab[u] = Ap + (int64_t)(8 * u + g) * K + 8 * WPT * t;
    }
    const float *sg = S + 2 * t;   // group sums of tokens 2t, 2t + 1 (+ 8u)
    auto load_ops = [&](int gi, uint4 (&o)[NT][WPT], float2 (&so)[NT]) {
#pragma unroll
        for (int u = 0; u < NT; ++u) {
            if (has[u]) {
#pragma unroll
                for (int i = 0; i < WPT; ++i) o[u][i] = ld_ro_v4(ab[u] + gi * GROUP + 8 * i);
            }
            so[u] = __ldg(reinterpret_cast<const float2 *>(sg + (int64_t)gi * TP + 8 * u));
        }
    };
    // operands of the current group (q, sq) and of the next one (n, sn)
    uint4 q[NT][WPT], n[NT][WPT];
    float2 sq[NT], sn[NT];
#pragma unroll
    for (int u = 0; u < NT; ++u) {
        sq[u] = sn[u] = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < WPT; ++i) q[u][i] = n[u][i] = make_uint4(0u, 0u, 0u, 0u);
    }
    if (nu > 0) load_ops(part * GS, q, sq);

    int j = 0;
    bool ok = true;
    uint32_t slot = 0, phase = 0;
    int st = part;   // current stage
#pragma unroll 1
    for (; j < nu; ++j) {
        if (!wait_bar_warp(bar0 + 8u * slot, phase, abort_flag, d_error)) {
            ok = false;
            break;
        }
        const uint32_t base = ring + slot * (uint32_t)L::SLOT;
        const float *tabc = tabw + (j & 1) * (L::TAB_STAGE / 4);
        const bool more = j + 1 < nu;
        const int st_next = st + P;
        if (more) sz_load(st_next, sr, zr);   // stored after this stage
#pragma unroll
        for (int h = 0; h < GS; ++h) {
            const int gi = st * GS + h;
            if (gi < G) {   // warp-uniform (the last stage may hold fewer groups)
                // the next group of this warp: the following one of this stage, else the first of its next stage
                const int gn = h + 1 < GS ? gi + 1 : st_next * GS;
                if (gn < G && (h + 1 < GS || more)) load_ops(gn, n, sn);
                uint32_t xa[R][WPT], xb[R][WPT];   // words of rows g and g + 8 of each block
#pragma unroll
                for (int b = 0; b < R; ++b) {
                    const uint32_t adr = base + (uint32_t)(b * 2048) + woff[h];
                    if constexpr (WPT == 4) {
                        const uint4 v = ptx::lds128(adr), w = ptx::lds128(adr + 1024u);
                        xa[b][0] = v.x;
                        xa[b][1 % WPT] = v.y;
                        xa[b][2 % WPT] = v.z;
                        xa[b][3 % WPT] = v.w;
                        xb[b][0] = w.x;
                        xb[b][1 % WPT] = w.y;
                        xb[b][2 % WPT] = w.z;
                        xb[b][3 % WPT] = w.w;
                    } else if constexpr (WPT == 2) {
                        asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(xa[b][0]), "=r"(xa[b][1 % WPT]) : "r"(adr));
                        asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];"
                                     : "=r"(xb[b][0]), "=r"(xb[b][1 % WPT])
                                     : "r"(adr + 1024u));
                    } else {
                        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(xa[b][0]) : "r"(adr));
                        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(xb[b][0]) : "r"(adr + 1024u));
                    }
                }
                float d0[R][NT][4], d1[R][NT][4];   // k-steps 2i and 2i + 1
#pragma unroll
                for (int i = 0; i < WPT; ++i) {
#pragma unroll
                    for (int b = 0; b < R; ++b) {
                        const uint32_t a00 = pair128(xa[b][i], 0), a01 = pair128(xb[b][i], 0),
                                       a02 = pair128(xa[b][i], 1), a03 = pair128(xb[b][i], 1);
                        const uint32_t a10 = pair128(xa[b][i], 2), a11 = pair128(xb[b][i], 2),
                                       a12 = pair128(xa[b][i], 3), a13 = pair128(xb[b][i], 3);
#pragma unroll
                        for (int u = 0; u < NT; ++u) {
                            if (i == 0) {
                                mma_first(d0[b][u], a00, a01, a02, a03, q[u][0].x, q[u][0].y);
                                mma_first(d1[b][u], a10, a11, a12, a13, q[u][0].z, q[u][0].w);
                            } else {
                                mma_acc(d0[b][u], a00, a01, a02, a03, q[u][i].x, q[u][i].y);
                                mma_acc(d1[b][u], a10, a11, a12, a13, q[u][i].z, q[u][i].w);
                            }
                        }
                    }
                }
                // acc += s D_g + c S_g: rows g (s, c = e.x, e.y) and g + 8 (e.z, e.w), tokens 2t, 2t + 1
#pragma unroll
                for (int b = 0; b < R; ++b) {
                    const float4 e = *reinterpret_cast<const float4 *>(tabc + h * (R * 32) + 4 * (b * 8 + g));
#pragma unroll
                    for (int u = 0; u < NT; ++u) {
                        acc[b][u][0] = fmaf(e.x, d0[b][u][0] + d1[b][u][0], fmaf(e.y, sq[u].x, acc[b][u][0]));
                        acc[b][u][1] = fmaf(e.x, d0[b][u][1] + d1[b][u][1], fmaf(e.y, sq[u].y, acc[b][u][1]));
                        acc[b][u][2] = fmaf(e.z, d0[b][u][2] + d1[b][u][2], fmaf(e.w, sq[u].x, acc[b][u][2]));
                        acc[b][u][3] = fmaf(e.z, d0[b][u][3] + d1[b][u][3], fmaf(e.w, sq[u].y, acc[b][u][3]));
                    }
                }
#pragma unroll
                for (int u = 0; u < NT; ++u) {
                    sq[u] = sn[u];
#pragma unroll
                    for (int i = 0; i < WPT; ++i) q[u][i] = n[u][i];
                }
            }
        }
        if (more) sz_store((j + 1) & 1, sr, zr);
        // every lane's reads of the slot have completed (their values were
        // used above): hand it back to the copy engine for unit j + slots;
        // the next unit's table is written
        __syncwarp();
        if (lane == 0 && !stall && j + kSlots < nu) {
            ptx::fence_proxy_async_smem();
            issue(j + kSlots);
        }
        if (++slot == kSlots) {
            slot = 0;
            phase ^= 1u;
        }
        st = st_next;
    }
    if (!ok && !stall) {
        // stages issued but not consumed land before the ring is reused
        const int end = min(nu, j + kSlots);
        for (int j2 = j; j2 < end; ++j2)
            wait_bar_drain(bar0 + 8u * (uint32_t)(j2 % kSlots), (uint32_t)(j2 / kSlots) & 1u);
    }
    if (x >= tiles) return;   // (all P warps of an idle group leave together)

    // the P parts of tile x, added in part order: each warp leaves its sums
    // [token][row] in its ring, the P warps meet at a named barrier, and warp p
    // of the group stores tokens p, p + P, ...
    float *mine = reinterpret_cast<float *>(smem + warp * kSlots * L::SLOT);
#pragma unroll
    for (int b = 0; b < R; ++b)
#pragma unroll
        for (int u = 0; u < NT; ++u)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                mine[(8 * u + 2 * t + (e & 1)) * RW + 16 * b + prow + 8 * (e >> 1)] = acc[b][u][e];
    if (P == 1) __syncwarp();
    else if (warp < P) asm volatile("bar.sync 1, %0;" ::"r"(32 * P) : "memory");   // the CTA's first group
    else asm volatile("bar.sync 2, %0;" ::"r"(32 * P) : "memory");                 // its second (P = 2)
    if (*abort_flag) return;
    const int nn = n0 + lane;   // lane = row of the tile
    const int w0 = warp - part;  // first warp of the group
    for (int tok = part; tok < M && tok < TP; tok += P) {
        float v = 0.f;
        for (int p2 = 0; p2 < P; ++p2)
            v += reinterpret_cast<const float *>(smem + (w0 + p2) * kSlots * L::SLOT)[tok * RW + lane];
        if (nn < N) C[(int64_t)tok * N + nn] = f32_to_bf16_rn(v);
    }
}

template <typename Kern, typename... Args>
cudaError_t launch_pdl(Kern kern, int grid, int block, int smem, cudaStream_t st, Args... args)
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

template <int NT, int WPT>
cudaError_t launch_frag_t(const CUtensorMap &m, const GemmArgs &a, const LaunchCtx &c, const uint16_t *Ap,
                          const float *S, int grid, int P)
{
    using L = FragLayout<NT, 8 / WPT>;
    auto kern = k_w4_frag<NT, WPT>;
    static std::once_flag once[64];
    static cudaError_t attr_err[64];
    int dev = 0;
    cudaGetDevice(&dev);
    std::call_once(once[dev & 63], [&] {
        attr_err[dev & 63] = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::BYTES);
    });
    if (attr_err[dev & 63] != cudaSuccess) return attr_err[dev & 63];
    return launch_pdl(kern, grid, kThreads, L::BYTES, c.stream, m, Ap, S, (const uint16_t *)a.scales,
                      (const uint8_t *)a.zeros, (uint16_t *)a.C, (int)a.M, (int)a.N, (int)a.K, P, c.d_error,
                      g_debug_stall);
}

template <int NT>
cudaError_t launch_frag_nt(const CUtensorMap &m, const GemmArgs &a, const LaunchCtx &c, const uint16_t *Ap,
                           const float *S, int grid, int P)
{
    switch (a.group) {
    case 32: return launch_frag_t<NT, 1>(m, a, c, Ap, S, grid, P);
    case 64: return launch_frag_t<NT, 2>(m, a, c, Ap, S, grid, P);
    default: return launch_frag_t<NT, 4>(m, a, c, Ap, S, grid, P);
    }
}

}  // namespace

// Warps per tile: the fewest (1, 2 or 4) that give at least three quarters
// of the device's resident warps work, and no more than there are stages.
int w4_frag_split(int64_t N, int64_t K, int sm_count, int tile_m)
{
    const int64_t tiles = (N + kW4FragRows - 1) / kW4FragRows, nst = (K + 255) / 256;
    const int64_t resident = (int64_t)sm_count * (tile_m <= 8 ? 4 : 2) * kW4FragWarps;
    int P = 1;
    while (P < kW4FragWarps && 2 * P <= nst && tiles * P * 4 < resident * 3) P *= 2;
    return P;
}
int w4_frag_grid(int64_t N, int P) { return (int)(((N + kW4FragRows - 1) / kW4FragRows * P + kW4FragWarps - 1) / kW4FragWarps); }

// Workspace, in floats: the activation copy (bf16 [M, K], 256-byte aligned
// end), then the group sums [G][tile_m].
int64_t w4_frag_workspace_floats(int64_t M, int64_t TP, int64_t K, int64_t group)
{
    return (M * K + 127) / 128 * 64 + TP * (K / group);
}

cudaError_t launch_w4_prep(const GemmArgs &a, const LaunchCtx &c, uint16_t *Ap, float *S, int TP)
{
    const int64_t items = (int64_t)TP * (a.K / 8);
    return launch_pdl(k_w4_frag_prep, (int)((items + 255) / 256), 256, 0, c.stream, (const uint16_t *)a.A, Ap, S,
                      (int)a.M, TP, (int)a.K, (int)a.group);
}

cudaError_t launch_w4_frag(const GemmArgs &a, const Plan &p, const LaunchCtx &c)
{
    if (!c.act_copy) return cudaErrorInvalidValue;
    const int TP = p.tile_m;
    uint16_t *Ap = (uint16_t *)c.act_copy;
    float *S = reinterpret_cast<float *>(Ap + (a.M * a.K + 127) / 128 * 128);
    CUtensorMap m;
    if (!make_map_words(&m, a.B, a.N, a.K, kW4FragRows)) return cudaErrorInvalidValue;
    cudaError_t e = launch_w4_prep(a, c, Ap, S, TP);
    if (e != cudaSuccess) return e;
    return TP <= 8 ? launch_frag_nt<1>(m, a, c, Ap, S, p.grid, p.split)
                   : launch_frag_nt<2>(m, a, c, Ap, S, p.grid, p.split);
}

}  // namespace dbw
