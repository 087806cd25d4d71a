// internal.h -- interface between the host API (api.cu) and the kernel
// translation units.  Not installed; not part of the C ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dbw_gemm.h"

namespace dbw {

// Per-call launch context built by the host API.
struct LaunchCtx {
    cudaStream_t stream;
    int sm_count;
    int *d_error;          // device error word (GEMM_ERR_DEVICE_TIMEOUT on a bounded-wait expiry)
    float *workspace;      // split-K partial tiles (fp32), may be null if the plan has split == 1
    int *counters;         // per-tile arrival counters, zero between calls
    int64_t ws_floats;     // capacity of `workspace` in floats
    int64_t n_counters;    // capacity of `counters`
    void *act_copy;        // W4A16 tcgen05: bf16 [M, K] activations in the kernel's k order (workspace)
};

struct GemmArgs {
    const void *A, *B;     // bf16 activations / bf16 weights (or packed int4 for W4A16)
    const void *scales, *zeros;
    void *C;
    int64_t M, N, K, lda, ldb, ldc, group;
    const void *bias = nullptr;   // bf16 [N] for GEMM_EPI_BIAS
    int epi = GEMM_EPI_NONE;      // bf16 only; for GEMM_EPI_SILU_MUL, N counts the columns of C and B has 2N rows
    const int *gends = nullptr;   // grouped GEMM: int32 cumulative token-row ends per expert (device)
    int64_t groups = 0;           //   experts; B is [groups, N, K]
    const void *sfa = nullptr;    // block-scaled GEMM: E8M0 scales of A [M, K/32] and B [N, K/32]
    const void *sfb = nullptr;
};

// Grouped GEMM: experts the prefill kernel's shared-memory table holds, and
// the (smaller) number the pair kernel's holds.
constexpr int kMaxExperts = 1024;
constexpr int kPairMaxExperts = 192;

// Host-side plan (pure function of the sizes and the SM count).
struct Plan {
    int variant;
    int kernels;
    int grid;
    int split;
    int tile_m, tile_n;
    int stages;
    int m_per_pass;        // GEMV: rows of A handled per pass over the weights
    int mode;              // tcgen05: 0 whole tiles round-robin, 1 stream-K, 2 cluster split-K
    int bn;                // tcgen05: MMA N (columns of the Y operand per tile)
    int group_r;           // tcgen05: tile-rows per raster group
    int ctas_per_sm;       // tcgen05 skinny: 1 = deep pipeline, 2 = shallow (two CTAs per SM)
    int whole = 0;         // tcgen05 mode 1: leading tiles done whole (the full waves), then stream-K
    int sk_grid = 0;       // tcgen05 mode 1: CTAs sharing the stream-K units (0 = all)
    int act_copy;          // W4A16: activations are first copied into the kernels' k order
    int64_t ws_extra;      // W4A16 register variant: fp32 group sums after the copy (floats)
};

// query = true: plan for the current device (asks it for cluster occupancy);
// false: host-only model of a device with sm_count SMs.
// pairs: the weight rows come in (gate, up) pairs (GEMM_EPI_SILU_MUL; N is
// then the kernel's row count 2 * columns of C): splits keep pairs together.
// fused: any epilogue (the pair kernel stores the plain product only).
bool plan_bf16(int64_t M, int64_t N, int64_t K, int variant, int sm_count, Plan *p, bool query = true,
               bool pairs = false, bool fused = false);
bool plan_w4a16(int64_t M, int64_t N, int64_t K, int64_t group, int variant, int sm_count, Plan *p,
                bool query = true);
// Grouped GEMM over G experts sharing M stacked token rows (prefill kernel,
// persistent whole tiles; the tile count is found on the device).
void plan_grouped(int64_t G, int64_t M, int64_t N, int64_t K, int sm_count, Plan *p);

// Workspace need (floats, counters) for a plan; 0 when it needs none.  The
// permuted activation copy of a W4A16 tcgen05 plan sits after the split-K
// partials, at float offset act_copy_offset(p).
void workspace_need(const Plan &p, int64_t M, int64_t N, int64_t K, int64_t *floats, int64_t *counters);
int64_t act_copy_offset(const Plan &p);

// Kernel launchers: return cudaSuccess or the launch error.
cudaError_t launch_zero_fill(const GemmArgs &a, const LaunchCtx &c);
cudaError_t launch_gemv_bf16(const GemmArgs &a, const Plan &p, const LaunchCtx &c);
cudaError_t launch_gemv_w4a16(const GemmArgs &a, const Plan &p, const LaunchCtx &c);
cudaError_t launch_umma_bf16(const GemmArgs &a, const Plan &p, const LaunchCtx &c);
// W4A16, M <= 32: dequantisation into mma.sync fragments (w4mma.cu); the
// kernel stages a CTA's scales and zeros in shared memory, up to this many
// groups per row
constexpr int kW4RegisterMaxGroups = 544;
cudaError_t launch_w4_register(const GemmArgs &a, const Plan &p, const LaunchCtx &c);
int w4_register_grid(int64_t N);
// W4A16, M <= 16: weights dequantised into mma.sync fragments, streamed by
// TMA (w4frag.cu): CTAs of kW4FragWarps warps; a tile of kW4FragRows weight
// rows is shared by w4_frag_split warps of a CTA.  The workspace holds the
// activation copy and the group sums (w4_frag_workspace_floats floats;
// tile_m = the MMAs' token count, 8 or 16).
constexpr int kW4FragRows = 32;
constexpr int kW4FragWarps = 4;
cudaError_t launch_w4_frag(const GemmArgs &a, const Plan &p, const LaunchCtx &c);
// W4A16 for up to 16 tokens (w4gemv.cu): a cluster of two CTAs of
// kW4GemvWarps warps per tile of kW4GemvRows weight rows, the warps splitting
// K; one kernel, no workspace.
constexpr int kW4GemvRows = 32;
constexpr int kW4GemvWarps = 4;
constexpr int kW4GemvMaxGroups = 192;   // K / group: the tile's scale and zero rows are staged whole
cudaError_t launch_w4_gemv(const GemmArgs &a, const Plan &p, const LaunchCtx &c);
int w4_gemv_grid(int64_t N);
int w4_frag_split(int64_t N, int64_t K, int sm_count, int tile_m);
int w4_frag_grid(int64_t N, int P);
int64_t w4_frag_workspace_floats(int64_t M, int64_t TP, int64_t K, int64_t group);
// The W4A16 activation pre-pass (w4frag.cu): Ap = A with every 8-k block in
// the order 0,4,1,5,2,6,3,7, and S[g][m] = sum of A[m, k] over group g for
// tokens m < TP (zero for m >= M).  TP * K / 8 threads.
cudaError_t launch_w4_prep(const GemmArgs &a, const LaunchCtx &c, uint16_t *Ap, float *S, int TP);
// W4A16 on tcgen05 with per-group accumulators (w4tc.cu): token tiles of bn
// (16, 32 or 64), 128-k stages, stream-K over (weight tile, stage) units.
int w4tc_stages(int bn);
cudaError_t launch_w4tc(const GemmArgs &a, const Plan &p, const LaunchCtx &c);
// bf16 decode for up to kBandMaxTokens tokens (gemvband.cu): CTA c streams
// weight rows [c N / grid, (c + 1) N / grid) (at most kBandMaxRows) through
// bulk copies into warp-level MMAs; no workspace.  plan_band is false when
// the shape does not fit (then another variant serves it).  Plan.bn holds
// the k per stage.
constexpr int kBandMaxRows = 64;
constexpr int kBandMaxTokens = 32;
bool plan_band(int64_t M, int64_t N, int64_t K, int sm_count, Plan *p);
cudaError_t launch_gemv_band(const GemmArgs &a, const Plan &p, const LaunchCtx &c);
// Prefill on CTA pairs (umma2.cu): 256 x 256 tiles, tcgen05.mma.cta_group::2;
// the grid is twice the number of pairs.
void plan_pair(int64_t M, int64_t N, int64_t K, int sm_count, Plan *p);
cudaError_t launch_umma_pair(const GemmArgs &a, const Plan &p, const LaunchCtx &c);
// W4A16 with many tokens: weights dequantised to bf16 into the workspace
// (act_copy, N * K bf16), then the pair GEMM.
cudaError_t launch_w4_pair(const GemmArgs &a, const Plan &p, const LaunchCtx &c);
// Block-scaled (MX) GEMM (mxgemm.cu): fmt 0 = E4M3 x E4M3, 1 = packed E2M1 x
// E2M1; k per stage (128 bytes of every row) and the workspace bytes of the
// rearranged scale chunks; the launch runs the scale pre-pass, then the GEMM.
int mx_stage_k(int fmt);
int64_t mx_sf_workspace_bytes(int64_t M, int64_t N, int64_t K, int fmt, int bn);
cudaError_t launch_mx(const GemmArgs &a, const Plan &p, const LaunchCtx &c, int fmt);
void plan_mx(int64_t M, int64_t N, int64_t K, int fmt, int sm_count, Plan *p);
// bf16 [rows, K] K-major (leading dimension ld, elements): TMA boxes of 64 k x
// box_rows rows, 128-byte swizzle, out-of-range elements read as zero.
bool make_map_bf16(CUtensorMap *m, const void *ptr, int64_t rows, int64_t K, int64_t ld, int box_rows);
// Bytes [rows, width] (fp8 / packed fp4 codes): boxes of 128 bytes x box_rows
// rows, 128-byte swizzle.
bool make_map_u8(CUtensorMap *m, const void *ptr, int64_t rows, int64_t width, int box_rows);
// bf16 [rows, K], K a multiple of 64, as [K / 64][rows][64]: boxes of
// box_kb 64-k blocks x box_rows rows (box_kb make_map_bf16 boxes in one copy).
bool make_map_kblocks(CUtensorMap *m, const void *ptr, int64_t rows, int64_t K, int64_t ld, int box_rows, int box_kb);
// C [rows, cols] bf16 for TMA stores of 32 x 32 boxes (64-byte swizzle) or of
// 32 rows x 16 columns (32-byte swizzle).
bool make_map_c32(CUtensorMap *m, void *C, int64_t rows, int64_t cols, int64_t ld);
bool make_map_c16(CUtensorMap *m, void *C, int64_t rows, int64_t cols, int64_t ld);
// A fused gate/up weight [2N, K] (gate rows, then up rows) as the 3-D view
// [N][2][K]: boxes of 64 k x 2 x box_pairs put gate and up row j next to each
// other in shared memory (128-byte swizzle).
bool make_map_pairs(CUtensorMap *m, const void *ptr, int64_t N, int64_t K, int64_t ld, int box_pairs);
// Packed 4-bit weights [rows, K/8] (uint32): boxes of 16 words (128 k) x
// box_rows rows, 64-byte swizzle.
bool make_map_words16(CUtensorMap *m, const void *ptr, int64_t rows, int64_t K, int box_rows);

// tcgen05 kernel geometry (umma.cu)
constexpr int kUmmaBM = 128;
constexpr int kUmmaBK = 64;
int umma_stages(int bn, bool skinny, bool deep);
// Resident clusters of the skinny kernel on the current device (-1 on failure).
int umma_cluster_capacity(int bn, bool deep, int cluster, bool w4 = false);
int umma_w4_stages(int bn);
cudaError_t launch_umma_w4a16(const GemmArgs &a, const Plan &p, const LaunchCtx &c);
// TMA map of packed 4-bit weights [rows, K/8] (uint32): 32-word x box_rows boxes, 128-byte swizzle.
bool make_map_words(CUtensorMap *m, const void *ptr, int64_t rows, int64_t K, int box_rows);
// The same weights (K a multiple of 256) as [K / 256][rows][32 words]: box_kb
// make_map_words boxes in one copy.
bool make_map_words_kblocks(CUtensorMap *m, const void *ptr, int64_t rows, int64_t K, int box_rows, int box_kb);
// W4A16 decode for up to kW4BandMaxTokens tokens on bands of weight rows
// (w4band.cu): CTA c streams rows [c N / grid, (c + 1) N / grid) (at most
// kW4BandMaxRows) over all of K, K / group at most kW4BandMaxGroups; no
// workspace.  Plan.bn holds the k per stage.
constexpr int kW4BandMaxRows = 48;
constexpr int kW4BandMaxTokens = 8;
constexpr int kW4BandMaxGroups = 192;
bool plan_w4_band(int64_t M, int64_t N, int64_t K, int64_t group, int sm_count, Plan *p);
cudaError_t launch_w4_band(const GemmArgs &a, const Plan &p, const LaunchCtx &c);
extern int g_debug_stall;   // test hook: producers issue no copies (forces the watchdog)

}  // namespace dbw
