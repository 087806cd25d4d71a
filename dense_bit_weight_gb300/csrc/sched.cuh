// sched.cuh -- the persistent tile schedule shared by the TMA-fed tcgen05
// kernels (umma.cu, w4tc.cu): whole tiles round-robin in a grouped raster,
// stream-K ranges of (tile, k-block) units with a deterministic last-arriver
// fixup, or one tile per CTA of a split-K cluster; and the bf16 stores of an
// output chunk.
//
// Stream-K (mode 1): the units of the tiles after the first `whole` ones are
// cut into sk_grid contiguous equal ranges, one per CTA.  A CTA stores the
// fp32 partial of a split tile in its workspace slot, bumps the tile's
// counter, and the last contributor adds every partial in increasing-k order
// (deterministic, no float atomics) and resets the counter to zero.
#pragma once

#include <stdint.h>

#include "common.cuh"

namespace dbw {

constexpr int kTileRows = 128;   // rows of X per tile (the MMA's M)

struct Sched {
    int mode;                    // 0 whole tiles, 1 stream-K ranges
    int tiles_r, tiles_q, tiles;
    int nk;                      // k-blocks per tile
    int grid;
    int group_r;                 // raster: tile-rows per group
    int stall;                   // test hook: producer issues nothing (forces the watchdog)
    int split;                   // mode 2: CTAs per tile (cluster size)
    long long units;             // mode 1: stream-K units, (tiles - whole) * nk
    int whole;                   // mode 1: leading tiles done whole, round-robin over the grid (the full waves)
    int sk_grid;                 // mode 1: CTAs sharing the stream-K units (<= grid)
    int epi;                     // fused epilogue (GEMM_EPI_*)
    int pairs;                   // the weight operand's map interleaves (gate, up) rows: 3-D copies
    const uint16_t *bias;        // GEMM_EPI_BIAS: bf16 per weight row (output column)
    const int *gends;            // grouped GEMM (prefill kernel, mode 0): cumulative token-row ends per expert
    int groups;                  //   experts
    int gN;                      //   weight rows per expert (columns of C)
    int tma_c;                   // mode 2: each CTA's block of the tile leaves through a TMA store (tmC)
    int x_bytes;                 // bytes one stage's X copy delivers (its box may be short: one token tile)
};


struct Segment {
    int tile, kb0, kb1, slot;
};

__device__ __forceinline__ void tile_coords(const Sched &s, int t, int &tr, int &tq)
{
    const int per_group = s.group_r * s.tiles_q;
    const int g = t / per_group;
    const int first_r = g * s.group_r;
    const int rows_in = min(s.group_r, s.tiles_r - first_r);
    const int local = t - g * per_group;
    tr = first_r + local % rows_in;
    tq = local / rows_in;
}

// Mode 1: first unit of CTA c's stream-K range (units of tiles >= whole; CTAs
// c >= sk_grid have an empty range).
__device__ __forceinline__ long long range_begin(const Sched &s, int c)
{
    const int cc = c < s.sk_grid ? c : s.sk_grid;
    return (long long)s.whole * s.nk + (long long)cc * s.units / s.sk_grid;
}

// CTA whose stream-K range contains unit u (mode 1).
__device__ __forceinline__ int cta_of_unit(const Sched &s, long long u)
{
    const long long v = u - (long long)s.whole * s.nk;
    return (int)(((v + 1) * s.sk_grid + s.units - 1) / s.units) - 1;
}

struct SegIter {
    long long u, u_end;
    int next_tile, count, sk;   // sk: stream-K segments so far (their workspace slot)
    int tiles;                  // mode 0: tiles to walk
    __device__ SegIter(const Sched &s, int cta, int ntiles) : tiles(ntiles)
    {
        count = 0;
        next_tile = cta;
        u = s.mode == 1 ? range_begin(s, cta) : 0;
        u_end = s.mode == 1 ? range_begin(s, cta + 1) : 0;
        sk = 0;
    }
    __device__ bool next(const Sched &s, Segment &seg)
    {
        if (s.mode == 2) {
            if (count > 0) return false;
            const int cta = next_tile;
            const int r = cta % s.split;
            seg.tile = cta / s.split;
            seg.kb0 = (int)((long long)r * s.nk / s.split);
            seg.kb1 = (int)((long long)(r + 1) * s.nk / s.split);
            seg.slot = 0;
        } else if (s.mode == 0) {
            if (next_tile >= tiles) return false;
            seg.tile = next_tile;
            seg.kb0 = 0;
            seg.kb1 = s.nk;
            seg.slot = 0;
            next_tile += s.grid;
        } else if (next_tile < s.whole) {   // mode 1: this CTA's whole tiles of the full waves first
            seg.tile = next_tile;
            seg.kb0 = 0;
            seg.kb1 = s.nk;
            seg.slot = 0;
            next_tile += s.grid;
        } else {
            if (u >= u_end) return false;
            seg.tile = (int)(u / s.nk);
            seg.kb0 = (int)(u % s.nk);
            const long long left = u_end - u;
            seg.kb1 = (int)min((long long)s.nk, seg.kb0 + left);
            seg.slot = sk == 0 ? 0 : 1;
            ++sk;
            u += seg.kb1 - seg.kb0;
        }
        ++count;
        return true;
    }
};

template <bool SWAP>
__device__ __forceinline__ void store_chunk(uint16_t *__restrict__ C, int64_t ldc, int R, int Q, int r,
                                            int q0, const float (&f)[16])
{
    if (r >= R) return;
    if (!SWAP) {
        uint16_t *dst = C + (int64_t)r * ldc + q0;
        if (q0 + 16 <= Q) {
            uint4 w0, w1;
            w0.x = pack_bf16x2_rn(f[0], f[1]);
            w0.y = pack_bf16x2_rn(f[2], f[3]);
            w0.z = pack_bf16x2_rn(f[4], f[5]);
            w0.w = pack_bf16x2_rn(f[6], f[7]);
            w1.x = pack_bf16x2_rn(f[8], f[9]);
            w1.y = pack_bf16x2_rn(f[10], f[11]);
            w1.z = pack_bf16x2_rn(f[12], f[13]);
            w1.w = pack_bf16x2_rn(f[14], f[15]);
            reinterpret_cast<uint4 *>(dst)[0] = w0;
            reinterpret_cast<uint4 *>(dst)[1] = w1;
        } else {
#pragma unroll
            for (int j = 0; j < 16; ++j)
                if (q0 + j < Q) dst[j] = f32_to_bf16_rn(f[j]);
        }
    } else {
#pragma unroll
        for (int j = 0; j < 16; ++j)
            if (q0 + j < Q) C[(int64_t)(q0 + j) * ldc + r] = f32_to_bf16_rn(f[j]);
    }
}


// Stream-K fixup of tile t by its last contributor: the fp32 partials of the
// CTAs c_first..c_last (workspace slot 2c + 0 for a CTA's first stream-K
// segment, 2c + 1 after; [column / 4][row] float4 layout, BN columns) are
// summed per column in increasing contributor (= increasing k) order and
// handed to emit(c0, f) sixteen columns at a time (f = columns c0..c0+15 of
// this thread's row).  INFL float4 loads are kept in flight per thread.
template <int BN, int INFL, typename Emit>
__device__ __forceinline__ void streamk_fixup(const Sched &sched, const float *__restrict__ ws, int t, int row,
                                              Emit &&emit)
{
    const int c_first = cta_of_unit(sched, (long long)t * sched.nk);
    const int c_last = cta_of_unit(sched, (long long)(t + 1) * sched.nk - 1);
    // CB4 float4 columns of BATCH contributors at a time (CB4 a divisor of
    // BN / 4 and a multiple of 4, since BN is a multiple of 16)
    constexpr int CB4 = INFL <= 4 || (BN / 4) % 8 ? 4 : (BN / 4) % 16 ? 8 : 16;
    static_assert((BN / 4) % CB4 == 0 && CB4 % 4 == 0, "fixup column batches tile BN");
    constexpr int BATCH = INFL / CB4 > 0 ? INFL / CB4 : 1;
    const float4 *wsv = reinterpret_cast<const float4 *>(ws);
#pragma unroll 1
    for (int cb = 0; cb < BN / 4; cb += CB4) {
        float4 a4[CB4];
#pragma unroll
        for (int j = 0; j < CB4; ++j) a4[j] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 1
        for (int cta0 = c_first; cta0 <= c_last; cta0 += BATCH) {
            float4 v[BATCH][CB4];
#pragma unroll
            for (int u = 0; u < BATCH; ++u) {
                const int cta = cta0 + u;
                if (cta <= c_last) {
                    const int first_tile = (int)(range_begin(sched, cta) / sched.nk);
                    const int slot = first_tile == t ? 0 : 1;
                    const float4 *p = wsv + (int64_t)(cta * 2 + slot) * (kTileRows * BN / 4) +
                                      (int64_t)cb * kTileRows + row;
#pragma unroll
                    for (int j = 0; j < CB4; ++j) v[u][j] = __ldcg(p + j * kTileRows);
                }
            }
#pragma unroll
            for (int u = 0; u < BATCH; ++u)
                if (cta0 + u <= c_last) {
#pragma unroll
                    for (int j = 0; j < CB4; ++j) {
                        a4[j].x += v[u][j].x;
                        a4[j].y += v[u][j].y;
                        a4[j].z += v[u][j].z;
                        a4[j].w += v[u][j].w;
                    }
                }
        }
#pragma unroll
        for (int j16 = 0; j16 < CB4 / 4; ++j16) {
            float f[16];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                f[4 * u] = a4[4 * j16 + u].x;
                f[4 * u + 1] = a4[4 * j16 + u].y;
                f[4 * u + 2] = a4[4 * j16 + u].z;
                f[4 * u + 3] = a4[4 * j16 + u].w;
            }
            emit(cb * 4 + j16 * 16, f);
        }
    }
}

}  // namespace dbw
