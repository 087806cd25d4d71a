// api.cu -- the C ABI: argument checks, launch planning, per-device state.
//
// Every precondition is checked on the host before anything is enqueued; a
// failed check returns its gemm_status and launches nothing.  There is no
// fallback path: a shape no kernel supports is an error.
#include <cuda_runtime.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <vector>

#include "internal.h"

namespace dbw {
int gemv_grid(int64_t N, int sm_count);
}

namespace {

using namespace dbw;

constexpr int kMaxDevices = 64;
constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;

struct StreamWorkspace {
    float *partials = nullptr;
    int *counters = nullptr;
    int64_t floats = 0, n_counters = 0;
};

struct DeviceState {
    bool ready = false;
    int sm_count = 0;
    int cc_major = 0, cc_minor = 0;
    int *d_error = nullptr;
    std::map<cudaStream_t, StreamWorkspace> ws;  // one workspace per stream
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

int cuda_status(cudaError_t e) { return e == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA; }

// Lazily set up the current device.  Allocates the error word (so it must not
// run inside stream capture).
int device_state(DeviceState **out, int *dev_out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return GEMM_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return GEMM_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceState &s = g_dev[dev];
    if (!s.ready) {
        cudaDeviceProp prop;
        if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return GEMM_ERR_CUDA;
        if (!(prop.major == 10 && prop.minor == 3)) return GEMM_ERR_ARCH;
        s.sm_count = prop.multiProcessorCount;
        s.cc_major = prop.major;
        s.cc_minor = prop.minor;
        if (cudaMalloc(&s.d_error, sizeof(int)) != cudaSuccess) return GEMM_ERR_CUDA;
        if (cudaMemset(s.d_error, 0, sizeof(int)) != cudaSuccess) return GEMM_ERR_CUDA;
        s.ready = true;
    }
    *out = &s;
    *dev_out = dev;
    return GEMM_OK;
}

// The split-K workspace of (device, stream), grown to at least the request.
// Growing frees the old buffers after synchronising the device, so the first
// split call of a given size class should come before any stream capture.
int stream_workspace(DeviceState &s, cudaStream_t st, int64_t floats, int64_t counters,
                     StreamWorkspace **out)
{
    std::lock_guard<std::mutex> lk(g_mu);
    StreamWorkspace &w = s.ws[st];
    if (w.floats < floats || w.n_counters < counters) {
        if (w.partials || w.counters) {
            if (cudaDeviceSynchronize() != cudaSuccess) return GEMM_ERR_CUDA;
            cudaFree(w.partials);
            cudaFree(w.counters);
            w = StreamWorkspace();
        }
        // round up so neighbouring shapes reuse the allocation
        int64_t f = std::max<int64_t>(floats, int64_t(1) << 20);
        int64_t c = std::max<int64_t>(counters, 4096);
        if (cudaMalloc(&w.partials, (size_t)f * sizeof(float)) != cudaSuccess ||
            cudaMalloc(&w.counters, (size_t)c * sizeof(int)) != cudaSuccess ||
            cudaMemset(w.counters, 0, (size_t)c * sizeof(int)) != cudaSuccess) {
            cudaFree(w.partials);   // (either may be null)
            cudaFree(w.counters);
            w = StreamWorkspace();
            return GEMM_ERR_CUDA;
        }
        w.floats = f;
        w.n_counters = c;
    }
    *out = &w;
    return GEMM_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool epi_needs_bias(int epi)
{
    return epi == GEMM_EPI_BIAS || epi == GEMM_EPI_BIAS_RELU || epi == GEMM_EPI_BIAS_SILU || epi == GEMM_EPI_BIAS_GELU;
}

bool overlaps(const void *a, int64_t abytes, const void *b, int64_t bbytes)
{
    uintptr_t a0 = (uintptr_t)a, b0 = (uintptr_t)b;
    return a0 < b0 + (uintptr_t)bbytes && b0 < a0 + (uintptr_t)abytes;
}

// Byte extent of a row-major [rows, cols] matrix with leading dimension ld.
int64_t extent(int64_t rows, int64_t cols, int64_t ld, int64_t elem)
{
    return rows == 0 ? 0 : ((rows - 1) * ld + cols) * elem;
}

int check_sizes(int64_t M, int64_t N, int64_t K)
{
    if (M < 0 || N < 0 || K < 0) return GEMM_ERR_SHAPE;
    if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return GEMM_ERR_SHAPE;
    if (K % 8) return GEMM_ERR_SHAPE;
    return GEMM_OK;
}

// w4: the W4A16 entry point; mx_fmt: the block-scaled entry points (0 E4M3,
// 1 E2M1), -1 otherwise.
int run(const GemmArgs &a, const Plan &p, cudaStream_t st, bool w4, int mx_fmt = -1)
{
    DeviceState *s = nullptr;
    int dev = 0;
    int rc = device_state(&s, &dev);
    if (rc) return rc;
    LaunchCtx c{};
    c.stream = st;
    c.sm_count = s->sm_count;
    c.d_error = s->d_error;
    int64_t nf = 0, nc = 0;
    workspace_need(p, a.M, a.N, a.K, &nf, &nc);
    if (nf > 0 || nc > 0) {
        StreamWorkspace *w = nullptr;
        rc = stream_workspace(*s, st, nf, nc, &w);
        if (rc) return rc;
        c.workspace = w->partials;
        c.counters = w->counters;
        c.ws_floats = w->floats;
        c.n_counters = w->n_counters;
        if (p.act_copy) c.act_copy = w->partials + act_copy_offset(p);
    }
    cudaError_t e = cudaSuccess;
    switch (p.variant) {
    case GEMM_VARIANT_ZERO: e = launch_zero_fill(a, c); break;
    case GEMM_VARIANT_GEMV: e = w4 ? launch_gemv_w4a16(a, p, c) : launch_gemv_bf16(a, p, c); break;
    case GEMM_VARIANT_BAND:
        if (mx_fmt >= 0 || a.gends) return GEMM_ERR_VARIANT;
        e = w4 ? launch_w4_band(a, p, c) : launch_gemv_band(a, p, c);
        break;
    case GEMM_VARIANT_REGISTER:
        if (!w4) return GEMM_ERR_VARIANT;
        e = launch_w4_register(a, p, c);
        break;
    case GEMM_VARIANT_FRAGMENT:
        if (!w4) return GEMM_ERR_VARIANT;
        e = p.mode == 1 ? launch_w4_gemv(a, p, c) : launch_w4_frag(a, p, c);
        break;
    case GEMM_VARIANT_GROUPWISE:
        if (!w4) return GEMM_ERR_VARIANT;
        e = launch_w4tc(a, p, c);
        break;
    case GEMM_VARIANT_BLOCK_SCALED:
        if (mx_fmt < 0) return GEMM_ERR_VARIANT;
        e = launch_mx(a, p, c, mx_fmt);
        break;
    case GEMM_VARIANT_PAIR:
        if (mx_fmt >= 0 || (w4 && (a.epi != GEMM_EPI_NONE || a.gends))) return GEMM_ERR_VARIANT;
        e = w4 ? launch_w4_pair(a, p, c) : launch_umma_pair(a, p, c);
        break;
    case GEMM_VARIANT_SKINNY:
    case GEMM_VARIANT_PREFILL:
        if (w4 && p.variant != GEMM_VARIANT_SKINNY) return GEMM_ERR_VARIANT;
        e = w4 ? launch_umma_w4a16(a, p, c) : launch_umma_bf16(a, p, c);
        break;
    default: return GEMM_ERR_VARIANT;
    }
    return cuda_status(e);
}

int sm_count_for_plan(int num_sms, int *out)
{
    if (num_sms > 0) {
        *out = num_sms;
        return GEMM_OK;
    }
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return GEMM_ERR_CUDA;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return GEMM_ERR_CUDA;
    *out = n;
    return GEMM_OK;
}

void to_public(const Plan &p, gemm_plan *out)
{
    out->variant = p.variant;
    out->kernels = p.kernels;
    out->grid = p.grid;
    out->split = p.split;
    out->tile_m = p.tile_m;
    out->tile_n = p.tile_n;
    out->stages = p.stages;
    out->reserved = p.m_per_pass;
}

}  // namespace

// ------------------------------------------------------------------ planning

namespace dbw {

// Resident clusters of size `cs` for the skinny kernel: the device's answer
// when planning for the current device, else an ideal-packing model.
static int64_t cluster_capacity(int bn, bool deep, int cs, int sm_count, bool query)
{
    if (query) {
        const int n = umma_cluster_capacity(bn, deep, cs);
        if (n >= 0) return n;
    }
    return (int64_t)(deep ? 1 : 2) * sm_count / cs;
}

// tcgen05 planning.
// Skinny (decode, swap AB): one 128-row weight tile per CTA with K split over
// a cluster of S CTAs (mode 2).  When the tiles fit one wave the deep form
// (one CTA per SM) takes the largest S <= 8 whose clusters are all resident at
// once without exceeding one CTA per SM; otherwise the shallow form (two CTAs
// per SM) runs every tile unsplit, all resident together, so the HBM stream
// is shared evenly.  Beyond two tiles per SM, deep stream-K (mode 1).
// Prefill: whole tiles round-robin (mode 0), min(tiles, SMs) CTAs, whenever the
// tiles fill at least half the SMs; stream-K (mode 1) below that.  Measured on
// GB300 over the fifteen prefill shapes, whole tiles were as fast or faster on
// every shape (1.3-1.4x at M = 1024: stream-K's fp32 fixup of a 128 x 256 tile
// costs more than the wave quantisation it removes); the M = 512 down
// projection (64 tiles) is 1.13x faster with stream-K spreading it over every SM.
static void plan_umma(int64_t M, int64_t N, int64_t K, bool swap, int bn, int sm_count, bool query,
                      Plan *p, bool pairs = false)
{
    const int64_t R = swap ? N : M, Q = swap ? M : N;
    const int64_t tiles_r = (R + kUmmaBM - 1) / kUmmaBM;
    const int64_t tiles_q = (Q + bn - 1) / bn;
    const int64_t tiles = tiles_r * tiles_q;
    const int64_t nk = (K + kUmmaBK - 1) / kUmmaBK;
    const int64_t G = sm_count;
    p->variant = swap ? GEMM_VARIANT_SKINNY : GEMM_VARIANT_PREFILL;
    p->bn = bn;
    p->tile_m = swap ? bn : kUmmaBM;
    p->tile_n = swap ? kUmmaBM : bn;
    p->group_r = swap ? (int)tiles_r : (int)std::min<int64_t>(tiles_r, 16);
    p->kernels = 1;
    p->ctas_per_sm = 1;
    if (swap && tiles <= G) {
        int64_t S = 1;
        // (gate, up) row pairs: each CTA of a cluster reduces a block of rows
        // of the tile, so the split must divide 128 into even blocks
        for (int64_t s = 2; s <= 8 && s <= nk && tiles * s <= G; ++s)
            if ((!pairs || (s & (s - 1)) == 0) && cluster_capacity(bn, true, (int)s, sm_count, query) >= tiles)
                S = s;
        p->mode = 2;
        p->split = (int)S;
        p->grid = (int)(tiles * S);
        p->stages = umma_stages(bn, true, true);
        return;
    }
    if (swap && tiles <= 2 * G) {
        p->mode = 2;
        p->split = 1;
        p->grid = (int)tiles;
        p->ctas_per_sm = 2;
        p->stages = umma_stages(bn, true, false);
        return;
    }
    p->stages = umma_stages(bn, swap, true);
    const int64_t rem = tiles % G;   // tiles of a last, partial wave
    if (!swap && tiles > G && rem * 4 > G && rem * 2 <= G && !pairs) {
        // full waves of whole tiles, then each leftover tile split along K
        // among S = 2 or 3 CTAs so the last wave ends after 1/S of a tile's
        // time.  Measured on the prefill sweep: a leftover of a quarter to half
        // a wave gains (1024 x 6144: +6%, 4096 x 4096 x 12288: +7%); smaller
        // leftovers split four ways lose more in the fixup than they save
        // (4096 x 24576: -4%) and stay whole tiles.
        const int64_t S = std::min<int64_t>({3, G / rem, nk});
        p->mode = 1;
        p->grid = (int)G;
        p->whole = (int)(tiles - rem);
        p->sk_grid = (int)(rem * S);
        p->split = (int)S;
    } else if (!swap && 2 * tiles >= G) {
        p->mode = 0;
        p->grid = (int)std::min<int64_t>(tiles, G);
        p->split = 1;
    } else {
        const int64_t units = tiles * nk;
        p->mode = 1;
        p->grid = (int)std::min<int64_t>(G, units);
        if (!swap && tiles_r > 1 && p->grid >= 2 * tiles_r) {
            // token tiles in lockstep: tile-rows in order (group_r = 1) and a
            // grid that is a multiple of them, so CTA c and CTA c + grid / tiles_r
            // cover the same (weight tile, k) units of neighbouring token tiles
            // at the same time and each weight stage comes from HBM once
            p->grid = p->grid / (int)tiles_r * (int)tiles_r;
            p->group_r = 1;
        }
        const int64_t per_cta = units / p->grid;   // >= 1
        p->split = (int)std::min<int64_t>(p->grid, (nk + per_cta - 1) / per_cta + 1);
        if (p->split < 1) p->split = 1;
    }
}

// Weight-tile width of the prefill kernel when the tokens fit one 128-row
// MMA tile: the weights are then read by exactly one CTA each, and the
// narrowest width (of the compiled ones) whose tiles fit one wave puts the
// most SMs on the stream.  0 when no such plan suits the shape: the tiles would
// fill less than 85% of the SMs, or a CTA's activations (M rows) would
// outweigh its weights (bn rows), which the split-K skinny kernel avoids.
// Measured on GB300 at N = 24576, K = 4096 against the skinny kernel's 192
// tiles of 128 weight rows, two CTAs on some SMs: 176-row tiles on 140 SMs
// take 34.2 us instead of 40.5 at M = 128, 32.7 instead of 35.7 at M = 64 and
// 32.2 instead of 33.9 at M = 32, 32.7 instead of 33.0 at M = 8 (the
// activation copies then cover the token rows only) and 32.6 against the
// GEMV's 33.6 at M = 1.  The fused gate/up pairs gain only from M = 64 on
// (M = 128: 4.95 TB/s against the skinny kernel's 4.0; M = 32: 4.98 against
// 5.5, M = 8: 4.95 against 5.9).
static int wide_bn(int64_t M, int64_t N, int sm_count, bool pairs)
{
    if (M > kUmmaBM || (pairs && M < 64)) return 0;
    for (int bn : {176, 192, 224, 256}) {
        const int64_t tiles = (N + bn - 1) / bn;
        if (tiles > sm_count) continue;
        if (tiles * 100 < 85LL * sm_count || bn < M) return 0;
        return bn;
    }
    return 0;
}

// Whether the band kernel (gemvband.cu) serves a decode shape under AUTO.
// Measured on GB300, graph-timed with the weights from HBM (us, band against
// the route it replaces): 6144 x 4096: M = 1 11.0 / 13.1 (GEMV), M = 4
// 11.0 / 26.5 (GEMV), M = 8 11.0 / 12.5 (skinny); 7168 x 4096: 11.3 / 14.0,
// 11.3 / 27.2, 11.2 / 13.2; 4096 x 4096 (27-row bands): M = 1 8.6 / 8.2,
// M = 4 8.6 / 14.9, M = 8 8.6 / 9.5; 4096 x 12288: M = 1 20.5 / 19.6,
// M = 4 20.5 / 38.8, M = 8 20.6 / 18.8; at M = 16 and 32 the skinny kernel
// leads (its tensor-core MMAs; the band kernel's warp-level ones grow with
// the tokens).  So: 2 to 4 tokens whenever a band fits; 1 and 5-8 tokens with
// K up to 8192, and at 1 token only bands of at least 32 rows.
static bool band_first(int64_t M, int64_t N, int64_t K, int sm_count, bool pairs)
{
    if (pairs || M > 8 || N < 1) return false;
    const int64_t rows = (N + std::min<int64_t>(sm_count, N) - 1) / std::min<int64_t>(sm_count, N);
    if (rows > kBandMaxRows) return false;
    if (M >= 2 && M <= 4) return true;
    return K <= 8192 && (M > 1 || rows >= 32);
}

bool plan_bf16(int64_t M, int64_t N, int64_t K, int variant, int sm_count, Plan *p, bool query, bool pairs,
               bool fused)
{
    *p = Plan{};
    if (K == 0) {
        if (variant != GEMM_VARIANT_AUTO && variant != GEMM_VARIANT_ZERO) return false;
        p->variant = GEMM_VARIANT_ZERO;
        p->kernels = 1;
        p->split = 1;
        return true;
    }
    if (variant == GEMM_VARIANT_AUTO) {
        // CTA pairs (256 x 256 tiles, cta_group::2) whenever their tiles keep
        // at least half the SM pairs busy: measured on the fifteen prefill
        // shapes at 1185-1961 TFLOP/s against 1039-1683 for single-CTA
        // 128 x 256 tiles (every shape faster); below that the single-CTA
        // kernel's stream-K spreads the work over every SM
        const int64_t pair_tiles = ((M + 255) / 256) * ((N + 255) / 256);
        variant = M > 128 && 4 * pair_tiles >= sm_count                     ? GEMM_VARIANT_PAIR
                  : M > 128 || wide_bn(M, N, sm_count, pairs)               ? GEMM_VARIANT_PREFILL
                  : band_first(M, N, K, sm_count, pairs)                    ? GEMM_VARIANT_BAND
                  : M <= 4                                                  ? GEMM_VARIANT_GEMV
                                                                            : GEMM_VARIANT_SKINNY;
    }
    switch (variant) {
    case GEMM_VARIANT_GEMV:
        p->variant = GEMM_VARIANT_GEMV;
        p->kernels = 1;
        p->split = 1;
        p->m_per_pass = (int)std::min<int64_t>(M, 4);
        p->tile_m = p->m_per_pass;
        p->tile_n = 8;
        p->grid = gemv_grid(pairs ? N / 2 : N, sm_count);   // pairs: one warp per (gate, up) row pair
        return true;
    case GEMM_VARIANT_SKINNY: {
        if (M > 128) return false;
        int bn = 16;
        while (bn < M) bn *= 2;
        plan_umma(M, N, K, true, bn, sm_count, query, p, pairs);
        return true;
    }
    case GEMM_VARIANT_PREFILL: {
        const int bn = wide_bn(M, N, sm_count, pairs);
        plan_umma(M, N, K, false, bn ? bn : 256, sm_count, query, p, pairs);
        return true;
    }
    case GEMM_VARIANT_BAND:
        // the (gate, up) pairs of the SiLU-mul epilogue are not served here
        return !pairs && plan_band(M, N, K, sm_count, p);
    case GEMM_VARIANT_PAIR: {
        (void)fused;   // every epilogue runs on the pair kernel (N: weight rows, 2N for (gate, up) pairs)
        p->variant = GEMM_VARIANT_PAIR;
        p->kernels = 1;
        p->bn = 256;
        p->tile_m = 256;
        p->tile_n = 256;
        p->stages = 6;
        p->ctas_per_sm = 1;
        plan_pair(M, N, K, sm_count, p);
        return true;
    }
    default: return false;
    }
}

void plan_grouped(int64_t G, int64_t M, int64_t N, int64_t K, int sm_count, Plan *p)
{
    *p = Plan{};
    p->variant = GEMM_VARIANT_PREFILL;
    p->kernels = 1;
    p->bn = 256;
    p->tile_m = kUmmaBM;
    p->tile_n = 256;
    p->mode = 0;
    p->split = 1;
    p->ctas_per_sm = 1;
    p->stages = umma_stages(256, false, true);
    // at most one partial m-tile per expert beyond the M / BM full ones
    const int64_t tiles = ((M + kUmmaBM - 1) / kUmmaBM + G) * ((N + 255) / 256);
    p->grid = (int)std::max<int64_t>(1, std::min<int64_t>(tiles, sm_count));
    p->group_r = 1;
    (void)K;
    if (G <= kPairMaxExperts && M >= 256 * G) {
        // experts of at least 256 tokens on average: CTA pairs with 256-row
        // m-tiles (an expert's last, partial one stores its rows directly)
        const int64_t pt = ((M + 255) / 256 + G) * ((N + 255) / 256);
        p->variant = GEMM_VARIANT_PAIR;
        p->tile_m = 256;
        p->stages = 6;
        p->grid = (int)(2 * std::max<int64_t>(1, std::min<int64_t>(pt, sm_count / 2)));
    }
}

// W4A16 routing (AUTO), from GB300 timings over the four decode shapes
// (N, K) in {(7168, 5120), (5120, 5120), (34816, 5120), (5120, 17408)}:
//   M <= 16, at most three CTAs per SM (two per 32-row tile)
//                fragment kernel with K split over clusters of two CTAs
//                (w4gemv.cu, mode 1): M = 1: 9.4 / 8.8 / - / 22.5 us, M = 8:
//                10.0 / 9.2 / - / 23.5, M = 16: 13.3 / 12.4 / - / 29.3, against
//                11.1 / 11.0 / - / 30.3 (M = 1) for the fragment kernel with a
//                pre-pass and 17.2 / 14.9 / - / 30.0 (M = 16) for tcgen05
//   M <= 8, more tiles
//                fragment kernel with a pre-pass (w4frag.cu, mode 0), its
//                warps resident at once: 31.7 us on 34816 x 5120 against 36.9
//                for the clusters running in waves
//   9 and up     tcgen05 kernel with in-kernel dequantisation into TMEM
//                (stages of 256 k, tokens in tiles of up to 128): cluster
//                split-K (mode 2) when the tiles fit one wave, stream-K
//                (mode 1) beyond; at M = 16 it leads the fragment kernel (44
//                vs 52 us on 34816 x 5120), whose activation loads grow with
//                M.  Above 128 tokens every weight tile is dequantised once
//                per token tile; the token tiles of a weight tile are
//                neighbours in the tile order, so its packed weights come
//                from L2 after the first.
bool plan_w4a16(int64_t M, int64_t N, int64_t K, int64_t group, int variant, int sm_count, Plan *p, bool query)
{
    *p = Plan{};
    if (K == 0) return false;
    if (variant == GEMM_VARIANT_AUTO) {
        // From 1024 tokens on, dequantise the weights once (2.5 bytes per
        // weight) and run the pair GEMM, when its waves of pair tiles are at
        // least three quarters full.  Measured on GB300 (fraction of the bf16
        // roofline, pair against the in-kernel dequantisation): 4096 x 34816
        // x 5120 0.875 against 0.546, 4096 x 5120 x 17408 0.779 against 0.466,
        // 2048 x 7168 x 5120 0.773 against 0.483, 1024 x 34816 x 5120 0.582
        // against 0.547; 1024 x 5120 x 17408 (80 pair tiles on 76 pairs: two
        // waves, the second almost empty) 0.439 against 0.477.
        const int64_t pair_tiles = ((M + 255) / 256) * ((N + 255) / 256);
        const int64_t pairs_n = std::max<int64_t>(1, sm_count / 2);
        const int64_t waves = (pair_tiles + pairs_n - 1) / pairs_n;
        const bool gemv_fits = 2 * ((N + kW4GemvRows - 1) / kW4GemvRows) <= 3 * (int64_t)sm_count &&
                               K / group <= kW4GemvMaxGroups;
        variant = M >= 1024 && 4 * pair_tiles >= 3 * waves * pairs_n ? GEMM_VARIANT_PAIR
                  : M <= 16 && gemv_fits                                ? GEMM_VARIANT_FRAGMENT
                  : M <= 8                                              ? GEMM_VARIANT_FRAGMENT
                                                                        : GEMM_VARIANT_SKINNY;
    }
    if (variant == GEMM_VARIANT_BAND) return plan_w4_band(M, N, K, group, sm_count, p);
    if (variant == GEMM_VARIANT_PAIR) {
        p->variant = GEMM_VARIANT_PAIR;
        p->kernels = 2;                      // dequantisation, then the pair GEMM
        p->act_copy = 1;
        p->ws_extra = N * K / 2;             // bf16 [N, K] as floats
        p->bn = 256;
        p->tile_m = 256;
        p->tile_n = 256;
        p->stages = 6;
        p->ctas_per_sm = 1;
        plan_pair(M, N, K, sm_count, p);
        return true;
    }
    if (variant == GEMM_VARIANT_REGISTER) {
        if (M > 32 || K / group > kW4RegisterMaxGroups) return false;
        p->variant = GEMM_VARIANT_REGISTER;
        p->kernels = 2;                      // activation copy and group sums, then the GEMM
        p->act_copy = 1;
        p->ws_extra = 32 * (K / group);   // group sums, tokens padded to the MMAs' 8, 16 or 32
        p->split = 1;
        p->m_per_pass = M <= 8 ? 1 : M <= 16 ? 2 : 4;   // MMAs of 8 tokens
        p->tile_m = 8 * p->m_per_pass;
        p->tile_n = 16;
        p->grid = w4_register_grid(N);
        return true;
    }
    if (variant == GEMM_VARIANT_GROUPWISE) {
        // tokens in tiles of 16, 32 or 64 (group 32: at most 32, the kernel's
        // eight per-group accumulators must fit beside its stage buffers);
        // 128-k stages; stream-K over every SM
        int bn = 16;
        while (bn < M && bn < (group == 32 ? 32 : 64)) bn *= 2;
        const int64_t tiles_r = (N + kUmmaBM - 1) / kUmmaBM, tiles_q = (M + bn - 1) / bn;
        const int64_t nk = (K + 127) / 128;
        const int64_t units = tiles_r * tiles_q * nk;
        p->variant = GEMM_VARIANT_GROUPWISE;
        p->kernels = 2;                      // activation copy and group sums, then the GEMM
        p->act_copy = 1;
        p->bn = bn;
        p->tile_m = bn;
        p->tile_n = kUmmaBM;
        p->group_r = tiles_q > 1 ? 1 : (int)tiles_r;   // token tiles of a weight tile run next to each other
        p->ctas_per_sm = 1;
        p->stages = w4tc_stages(bn);
        p->mode = 1;
        p->grid = (int)std::min<int64_t>(sm_count, units);
        const int64_t per_cta = units / p->grid;
        p->split = (int)std::min<int64_t>(p->grid, (nk + per_cta - 1) / per_cta + 1);
        p->ws_extra = tiles_q * bn * (K / group);   // group sums [K / group][tokens padded to whole tiles]
        return true;
    }
    if (variant == GEMM_VARIANT_FRAGMENT) {
        if (M > 16) return false;
        p->variant = GEMM_VARIANT_FRAGMENT;
        p->tile_m = M <= 8 ? 8 : 16;         // tokens of the MMAs (N side)
        const int64_t tiles = (N + kW4GemvRows - 1) / kW4GemvRows;
        if (2 * tiles <= 3 * (int64_t)sm_count && K / group <= kW4GemvMaxGroups) {
            // mode 1 (w4gemv.cu): a cluster of two CTAs per 32-row tile, all
            // resident at once; one kernel, no workspace
            p->mode = 1;
            p->kernels = 1;
            p->tile_n = kW4GemvRows;
            p->grid = w4_gemv_grid(N);
            p->split = (int)std::min<int64_t>(2 * kW4GemvWarps, (K + 127) / 128);   // warps sharing a tile's K
            return true;
        }
        // mode 0 (w4frag.cu): the activation pre-pass, then 32-row tiles
        // shared by 1, 2 or 4 warps of a CTA
        p->mode = 0;
        p->kernels = 2;
        p->act_copy = 1;
        p->tile_n = kW4FragRows;
        p->split = w4_frag_split(N, K, sm_count, p->tile_m);   // warps per tile
        p->grid = w4_frag_grid(N, p->split);
        p->ws_extra = w4_frag_workspace_floats(M, p->tile_m, K, group);   // activation copy and group sums
        return true;
    }
    if (variant == GEMM_VARIANT_SKINNY) {
        int bn = 16;
        while (bn < M && bn < 128) bn *= 2;
        const int64_t tiles_r = (N + kUmmaBM - 1) / kUmmaBM, tiles_q = (M + bn - 1) / bn;
        const int64_t tiles = tiles_r * tiles_q;
        const int64_t nk = (K + 4 * kUmmaBK - 1) / (4 * kUmmaBK);   // 256-k stages
        const int64_t G = sm_count;
        p->variant = GEMM_VARIANT_SKINNY;
        p->kernels = 2;                      // activation k-order copy, then the GEMM
        p->act_copy = 1;
        p->bn = bn;
        p->tile_m = bn;
        p->tile_n = kUmmaBM;
        p->group_r = tiles_q > 1 ? 1 : (int)tiles_r;   // token tiles of a weight tile run next to each other
        p->ctas_per_sm = 1;
        p->stages = umma_w4_stages(bn);
        if (tiles <= G) {
            int64_t S = 1;
            for (int64_t s = 2; s <= 8 && s <= nk && tiles * s <= G; ++s) {
                int64_t cap = (int64_t)sm_count / s;
                if (query) {
                    const int n = umma_cluster_capacity(bn, true, (int)s, true);
                    if (n >= 0) cap = n;
                }
                if (cap >= tiles) S = s;
            }
            p->mode = 2;
            p->split = (int)S;
            p->grid = (int)(tiles * S);
        } else {
            const int64_t units = tiles * nk;
            p->mode = 1;
            p->grid = (int)std::min<int64_t>(G, units);
            const int64_t per_cta = units / p->grid;
            p->split = (int)std::min<int64_t>(p->grid, (nk + per_cta - 1) / per_cta + 1);
        }
        return true;
    }
    if (variant != GEMM_VARIANT_GEMV) return false;
    p->variant = GEMM_VARIANT_GEMV;
    p->kernels = 1;
    p->split = 1;
    p->m_per_pass = M >= 4 ? 4 : (M >= 2 ? 2 : 1);
    p->tile_m = p->m_per_pass;
    p->tile_n = 8;
    p->grid = gemv_grid(N, sm_count);
    return true;
}

// Block-scaled GEMM: tiles of 128 rows of A x 256 rows of B (128 when N <=
// 128), stages of 128 bytes of every row.  Whole tiles round-robin when they
// fill at least half the SMs, stream-K over every SM below that.
void plan_mx(int64_t M, int64_t N, int64_t K, int fmt, int sm_count, Plan *p)
{
    *p = Plan{};
    if (K == 0) {
        p->variant = GEMM_VARIANT_ZERO;
        p->kernels = 1;
        p->split = 1;
        return;
    }
    const int bn = N <= 128 ? 128 : 256;
    const int64_t tiles_r = (M + kUmmaBM - 1) / kUmmaBM, tiles_q = (N + bn - 1) / bn;
    const int64_t tiles = tiles_r * tiles_q;
    const int64_t kst = mx_stage_k(fmt);
    const int64_t nk = (K + kst - 1) / kst;
    const int64_t G = sm_count;
    p->variant = GEMM_VARIANT_BLOCK_SCALED;
    p->kernels = 2;                          // scale rearrangement, then the GEMM
    p->act_copy = 1;
    p->bn = bn;
    p->tile_m = kUmmaBM;
    p->tile_n = bn;
    p->stages = 4;
    p->ctas_per_sm = 1;
    p->group_r = (int)std::min<int64_t>(tiles_r, 16);
    p->ws_extra = (mx_sf_workspace_bytes(M, N, K, fmt, bn) + 3) / 4;
    if (2 * tiles >= G) {
        p->mode = 0;
        p->grid = (int)std::min<int64_t>(tiles, G);
        p->split = 1;
    } else {
        const int64_t units = tiles * nk;
        p->mode = 1;
        p->grid = (int)std::min<int64_t>(G, units);
        const int64_t per_cta = units / p->grid;
        p->split = (int)std::min<int64_t>(p->grid, (nk + per_cta - 1) / per_cta + 1);
    }
}

// CTAs of a stream-K plan that write fp32 partial tiles: those sharing the
// stream-K units (CTA c keeps two partial slots at 2c and 2c + 1).  When full
// waves of whole tiles come first, only the first sk_grid CTAs share units.
static int64_t partial_writers(const Plan &p)
{
    if (p.variant == GEMM_VARIANT_PAIR) return 2 * (int64_t)p.sk_grid;   // both CTAs of each sharing pair
    return p.whole > 0 && p.sk_grid > 0 ? std::min(p.sk_grid, p.grid) : p.grid;
}

// Plans whose kernel keeps stream-K partials (and tile counters) in the workspace.
static bool streamk_partials(const Plan &p)
{
    return (p.variant == GEMM_VARIANT_SKINNY || p.variant == GEMM_VARIANT_PREFILL ||
            p.variant == GEMM_VARIANT_GROUPWISE || p.variant == GEMM_VARIANT_BLOCK_SCALED ||
            p.variant == GEMM_VARIANT_PAIR) &&
           p.mode == 1;
}

// fp32 partial floats of a stream-K plan: two tile slots per writer; the pair
// kernel's writers are its CTAs (each keeps its 128 rows of a 256-row tile).
static int64_t partial_floats(const Plan &p)
{
    return partial_writers(p) * 2 * kUmmaBM * p.bn;
}

int64_t act_copy_offset(const Plan &p)
{
    const bool split = streamk_partials(p);
    const int64_t partials = split ? partial_floats(p) : 0;
    return (partials + 63) / 64 * 64;   // 256-byte aligned
}

void workspace_need(const Plan &p, int64_t M, int64_t N, int64_t K, int64_t *floats, int64_t *counters)
{
    *floats = 0;
    *counters = 0;
    if (streamk_partials(p)) {
        *floats = partial_floats(p);
        *counters = ((M + p.tile_m - 1) / p.tile_m) * ((N + p.tile_n - 1) / p.tile_n);
        if (p.variant == GEMM_VARIANT_PAIR) *counters *= 2;   // one per CTA half of a tile
    }
    if (p.variant == GEMM_VARIANT_FRAGMENT) {   // mode 0: activation copy and group sums; mode 1: none
        if (p.mode == 0) *floats = p.ws_extra;
        return;
    }
    if (p.variant == GEMM_VARIANT_BLOCK_SCALED) {   // rearranged scale chunks after the partials
        *floats = act_copy_offset(p) + p.ws_extra;
        return;
    }
    if (p.variant == GEMM_VARIANT_PAIR) {   // W4A16: the dequantised weights after the partials
        *floats = act_copy_offset(p) + p.ws_extra;
        return;
    }
    else if (p.act_copy) *floats = act_copy_offset(p) + (M * K + 127) / 128 * 64 + p.ws_extra;   // bf16 [M, K] (+ sums)
}

}  // namespace dbw

// ------------------------------------------------------------------ C ABI

extern "C" {

int gemm_bf16_ex(const void *A, const void *B, void *C, int64_t M, int64_t N, int64_t K,
                 int64_t lda, int64_t ldb, int64_t ldc, void *stream, int variant)
{
    int rc = check_sizes(M, N, K);
    if (rc) return rc;
    if (M == 0 || N == 0) return GEMM_OK;
    // K == 0: A and B are empty and never read; only C is checked
    if (!C || (K > 0 && (!A || !B))) return GEMM_ERR_NULL;
    if (ldc < N || ldc % 8 || (K > 0 && (lda < K || ldb < K || lda % 8 || ldb % 8))) return GEMM_ERR_LD;
    if (!aligned16(C) || (K > 0 && (!aligned16(A) || !aligned16(B)))) return GEMM_ERR_ALIGN;
    const int64_t cb = extent(M, N, ldc, 2);
    if (K > 0 && (overlaps(C, cb, A, extent(M, K, lda, 2)) || overlaps(C, cb, B, extent(N, K, ldb, 2))))
        return GEMM_ERR_ALIAS;
    DeviceState *s = nullptr;
    int dev = 0;
    rc = device_state(&s, &dev);
    if (rc) return rc;
    Plan p;
    if (!plan_bf16(M, N, K, variant, s->sm_count, &p)) return GEMM_ERR_VARIANT;
    GemmArgs a{A, B, nullptr, nullptr, C, M, N, K, lda, ldb, ldc, 0};
    return run(a, p, (cudaStream_t)stream, false);
}

int gemm_bf16(const void *A, const void *B, void *C, int64_t M, int64_t N, int64_t K,
              int64_t lda, int64_t ldb, int64_t ldc, void *stream)
{
    return gemm_bf16_ex(A, B, C, M, N, K, lda, ldb, ldc, stream, GEMM_VARIANT_AUTO);
}

int gemm_bf16_fused_ex(const void *A, const void *B, const void *bias, void *C, int64_t M, int64_t N,
                       int64_t K, int64_t lda, int64_t ldb, int64_t ldc, int epilogue, void *stream,
                       int variant)
{
    if (epilogue < GEMM_EPI_NONE || epilogue > GEMM_EPI_BIAS_GELU) return GEMM_ERR_EPILOGUE;
    if (epi_needs_bias(epilogue) != (bias != nullptr)) return GEMM_ERR_EPILOGUE;
    if (epilogue == GEMM_EPI_NONE) return gemm_bf16_ex(A, B, C, M, N, K, lda, ldb, ldc, stream, variant);
    int rc = check_sizes(M, N, K);
    if (rc) return rc;
    const bool pairs = epilogue == GEMM_EPI_SILU_MUL;
    const int64_t NB = pairs ? 2 * N : N;   // rows of B
    if (NB > kMaxDim) return GEMM_ERR_SHAPE;
    if (M == 0 || N == 0) return GEMM_OK;
    if (!C || (K > 0 && (!A || !B))) return GEMM_ERR_NULL;
    if (ldc < N || ldc % 8 || (K > 0 && (lda < K || ldb < K || lda % 8 || ldb % 8))) return GEMM_ERR_LD;
    if (!aligned16(C) || (K > 0 && (!aligned16(A) || !aligned16(B)))) return GEMM_ERR_ALIGN;
    if (bias && ((uintptr_t)bias & 1u)) return GEMM_ERR_ALIGN;
    const int64_t cb = extent(M, N, ldc, 2);
    if (K > 0 && (overlaps(C, cb, A, extent(M, K, lda, 2)) || overlaps(C, cb, B, extent(NB, K, ldb, 2))))
        return GEMM_ERR_ALIAS;
    if (bias && overlaps(C, cb, bias, N * 2)) return GEMM_ERR_ALIAS;
    DeviceState *s = nullptr;
    int dev = 0;
    rc = device_state(&s, &dev);
    if (rc) return rc;
    Plan p;
    if (!plan_bf16(M, NB, K, variant, s->sm_count, &p, true, pairs, true)) return GEMM_ERR_VARIANT;
    GemmArgs a{A, B, nullptr, nullptr, C, M, N, K, lda, ldb, ldc, 0, bias, epilogue};
    return run(a, p, (cudaStream_t)stream, false);
}

int gemm_bf16_grouped(const void *A, const void *B, void *C, const void *ends, int64_t G, int64_t M,
                      int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc, void *stream)
{
    int rc = check_sizes(M, N, K);
    if (rc) return rc;
    if (G < 1 || G > kMaxExperts || K == 0 || G * N > kMaxDim) return GEMM_ERR_SHAPE;
    if (M == 0 || N == 0) return GEMM_OK;
    if (!A || !B || !C || !ends) return GEMM_ERR_NULL;
    if (ldc < N || ldc % 8 || lda < K || ldb < K || lda % 8 || ldb % 8) return GEMM_ERR_LD;
    if (!aligned16(A) || !aligned16(B) || !aligned16(C) || ((uintptr_t)ends & 3u)) return GEMM_ERR_ALIGN;
    const int64_t cb = extent(M, N, ldc, 2);
    if (overlaps(C, cb, A, extent(M, K, lda, 2)) || overlaps(C, cb, B, extent(G * N, K, ldb, 2)) ||
        overlaps(C, cb, ends, G * 4))
        return GEMM_ERR_ALIAS;
    DeviceState *s = nullptr;
    int dev = 0;
    rc = device_state(&s, &dev);
    if (rc) return rc;
    Plan p;
    plan_grouped(G, M, N, K, s->sm_count, &p);
    GemmArgs a{A, B, nullptr, nullptr, C, M, N, K, lda, ldb, ldc, 0};
    a.gends = (const int *)ends;
    a.groups = G;
    return run(a, p, (cudaStream_t)stream, false);
}

int gemm_bf16_fused(const void *A, const void *B, const void *bias, void *C, int64_t M, int64_t N, int64_t K,
                    int64_t lda, int64_t ldb, int64_t ldc, int epilogue, void *stream)
{
    return gemm_bf16_fused_ex(A, B, bias, C, M, N, K, lda, ldb, ldc, epilogue, stream, GEMM_VARIANT_AUTO);
}

int gemm_w4a16_ex(const void *A, const void *Bq, const void *scales, const void *zeros, void *C,
                  int64_t M, int64_t N, int64_t K, int64_t group, void *stream, int variant)
{
    int rc = check_sizes(M, N, K);
    if (rc) return rc;
    if (N % 8) return GEMM_ERR_SHAPE;
    if (group != 32 && group != 64 && group != 128) return GEMM_ERR_GROUP;
    if (K % group) return GEMM_ERR_GROUP;
    if (K == 0) return GEMM_ERR_SHAPE;
    if (M == 0 || N == 0) return GEMM_OK;
    if (!A || !Bq || !scales || !zeros || !C) return GEMM_ERR_NULL;
    if (!aligned16(A) || !aligned16(Bq) || !aligned16(C) || ((uintptr_t)scales & 1u))
        return GEMM_ERR_ALIGN;
    const int64_t cb = M * N * 2;
    if (overlaps(C, cb, A, M * K * 2) || overlaps(C, cb, Bq, N * K / 2) ||
        overlaps(C, cb, scales, N * (K / group) * 2) || overlaps(C, cb, zeros, N * (K / group)))
        return GEMM_ERR_ALIAS;
    DeviceState *s = nullptr;
    int dev = 0;
    rc = device_state(&s, &dev);
    if (rc) return rc;
    Plan p;
    if (!plan_w4a16(M, N, K, group, variant, s->sm_count, &p)) return GEMM_ERR_VARIANT;
    GemmArgs a{A, Bq, scales, zeros, C, M, N, K, K, K / 8, N, group};
    return run(a, p, (cudaStream_t)stream, true);
}

int gemm_w4a16(const void *A, const void *Bq, const void *scales, const void *zeros, void *C,
               int64_t M, int64_t N, int64_t K, int64_t group, void *stream)
{
    return gemm_w4a16_ex(A, Bq, scales, zeros, C, M, N, K, group, stream, GEMM_VARIANT_AUTO);
}

static int gemm_mx_checked(const void *A, const void *SA, const void *B, const void *SB, void *C, int64_t M,
                           int64_t N, int64_t K, void *stream, int fmt)
{
    int rc = check_sizes(M, N, K);
    if (rc) return rc;
    if (K % 128 || N % 8) return GEMM_ERR_SHAPE;
    if (M == 0 || N == 0) return GEMM_OK;
    if (!C || (K > 0 && (!A || !B || !SA || !SB))) return GEMM_ERR_NULL;
    if (!aligned16(C) || (K > 0 && (!aligned16(A) || !aligned16(B) || ((uintptr_t)SA & 3u) || ((uintptr_t)SB & 3u))))
        return GEMM_ERR_ALIGN;
    const int64_t cb = M * N * 2, eb = fmt == 0 ? K : K / 2;
    if (K > 0 && (overlaps(C, cb, A, M * eb) || overlaps(C, cb, B, N * eb) || overlaps(C, cb, SA, M * (K / 32)) ||
                  overlaps(C, cb, SB, N * (K / 32))))
        return GEMM_ERR_ALIAS;
    DeviceState *s = nullptr;
    int dev = 0;
    rc = device_state(&s, &dev);
    if (rc) return rc;
    Plan p;
    plan_mx(M, N, K, fmt, s->sm_count, &p);
    GemmArgs a{A, B, nullptr, nullptr, C, M, N, K, K, K, N, 0};
    a.sfa = SA;
    a.sfb = SB;
    return run(a, p, (cudaStream_t)stream, false, fmt);
}

int gemm_mxfp8(const void *A, const void *SA, const void *B, const void *SB, void *C, int64_t M, int64_t N, int64_t K,
               void *stream)
{
    return gemm_mx_checked(A, SA, B, SB, C, M, N, K, stream, 0);
}

int gemm_mxfp4(const void *A, const void *SA, const void *B, const void *SB, void *C, int64_t M, int64_t N, int64_t K,
               void *stream)
{
    return gemm_mx_checked(A, SA, B, SB, C, M, N, K, stream, 1);
}

int gemm_mx_plan(int64_t M, int64_t N, int64_t K, int fmt, int num_sms, gemm_plan *out)
{
    if (!out) return GEMM_ERR_NULL;
    int rc = check_sizes(M, N, K);
    if (rc) return rc;
    if (K % 128 || N % 8 || (fmt != 0 && fmt != 1)) return GEMM_ERR_SHAPE;
    int sms = 0;
    rc = sm_count_for_plan(num_sms, &sms);
    if (rc) return rc;
    Plan p;
    plan_mx(M, N, K, fmt, sms, &p);
    to_public(p, out);
    return GEMM_OK;
}

int gemm_bf16_plan(int64_t M, int64_t N, int64_t K, int variant, int num_sms, gemm_plan *out)
{
    if (!out) return GEMM_ERR_NULL;
    int rc = check_sizes(M, N, K);
    if (rc) return rc;
    int sms = 0;
    rc = sm_count_for_plan(num_sms, &sms);
    if (rc) return rc;
    Plan p;
    if (!plan_bf16(M, N, K, variant, sms, &p, num_sms == 0)) return GEMM_ERR_VARIANT;
    to_public(p, out);
    return GEMM_OK;
}

int gemm_bf16_fused_plan(int64_t M, int64_t N, int64_t K, int epilogue, int variant, int num_sms,
                         gemm_plan *out)
{
    if (epilogue < GEMM_EPI_NONE || epilogue > GEMM_EPI_BIAS_GELU) return GEMM_ERR_EPILOGUE;
    if (epilogue == GEMM_EPI_NONE) return gemm_bf16_plan(M, N, K, variant, num_sms, out);
    if (!out) return GEMM_ERR_NULL;
    int rc = check_sizes(M, N, K);
    if (rc) return rc;
    const bool pairs = epilogue == GEMM_EPI_SILU_MUL;
    const int64_t NB = pairs ? 2 * N : N;   // rows of B
    if (NB > kMaxDim) return GEMM_ERR_SHAPE;
    int sms = 0;
    rc = sm_count_for_plan(num_sms, &sms);
    if (rc) return rc;
    Plan p;
    if (!plan_bf16(M, NB, K, variant, sms, &p, num_sms == 0, pairs, true)) return GEMM_ERR_VARIANT;
    to_public(p, out);
    return GEMM_OK;
}

int gemm_w4a16_plan(int64_t M, int64_t N, int64_t K, int64_t group, int variant, int num_sms,
                    gemm_plan *out)
{
    if (!out) return GEMM_ERR_NULL;
    int rc = check_sizes(M, N, K);
    if (rc) return rc;
    if (group != 32 && group != 64 && group != 128) return GEMM_ERR_GROUP;
    if (K % group) return GEMM_ERR_GROUP;
    int sms = 0;
    rc = sm_count_for_plan(num_sms, &sms);
    if (rc) return rc;
    Plan p;
    if (!plan_w4a16(M, N, K, group, variant, sms, &p, num_sms == 0)) return GEMM_ERR_VARIANT;
    to_public(p, out);
    return GEMM_OK;
}

int gemm_last_device_error(void)
{
    DeviceState *s = nullptr;
    int dev = 0;
    int rc = device_state(&s, &dev);
    if (rc) return rc;
    int v = 0;
    if (cudaMemcpy(&v, s->d_error, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess)
        return GEMM_ERR_CUDA;
    if (v != 0 && cudaMemset(s->d_error, 0, sizeof(int)) != cudaSuccess) return GEMM_ERR_CUDA;
    return v;
}

const char *gemm_status_string(int status)
{
    switch (status) {
    case GEMM_OK: return "ok";
    case GEMM_ERR_NULL: return "a required pointer is NULL";
    case GEMM_ERR_SHAPE: return "unsupported or invalid shape";
    case GEMM_ERR_LD: return "invalid leading dimension";
    case GEMM_ERR_ALIGN: return "pointer not 16-byte aligned";
    case GEMM_ERR_GROUP: return "invalid W4A16 group size";
    case GEMM_ERR_CUDA: return "CUDA runtime error";
    case GEMM_ERR_DEVICE_TIMEOUT: return "device-side bounded wait expired";
    case GEMM_ERR_ARCH: return "device is not compute capability 10.3";
    case GEMM_ERR_ALIAS: return "output overlaps an input";
    case GEMM_ERR_VARIANT: return "variant cannot run this shape";
    case GEMM_ERR_EPILOGUE: return "unknown epilogue, or bias missing or not used";
    default: return "unknown status";
    }
}

int gemm_debug_inject_timeout(int enable)
{
    const int prev = dbw::g_debug_stall;
    dbw::g_debug_stall = enable ? 1 : 0;
    return prev;
}

void gemm_shutdown(void)
{
    std::lock_guard<std::mutex> lk(g_mu);
    int prev = -1;
    cudaGetDevice(&prev);
    for (int d = 0; d < kMaxDevices; ++d) {
        DeviceState &s = g_dev[d];
        if (!s.ready) continue;
        cudaSetDevice(d);
        cudaDeviceSynchronize();
        for (auto &kv : s.ws) {
            cudaFree(kv.second.partials);
            cudaFree(kv.second.counters);
        }
        s.ws.clear();
        cudaFree(s.d_error);
        s = DeviceState();
    }
    if (prev >= 0) cudaSetDevice(prev);
}

}  // extern "C"
