// Tile and k-range scheduling shared by the host planner and the kernels.
// Pure integer arithmetic, compiled for both host and device.
#pragma once

#include <cstdint>

#if defined(__CUDACC__)
#define TG_HD __host__ __device__ __forceinline__
#else
#define TG_HD inline
#endif

namespace tg {

// Persistent tile order: tiles are walked in groups of `group_m` row blocks;
// inside a group, down the rows first, then across the columns.  A wave of
// consecutive tile numbers therefore covers a group_m × (wave/group_m) block
// of C, whose A rows and B columns stay resident in L2 together.
struct TileCoord {
    int32_t m_blk;
    int32_t n_blk;
};

TG_HD TileCoord tile_coord(int32_t tile, int32_t tiles_m, int32_t tiles_n, int32_t group_m) {
    const int32_t per_group = group_m * tiles_n;
    const int32_t g = tile / per_group;
    const int32_t first_m = g * group_m;
    const int32_t rows_left = tiles_m - first_m;
    const int32_t gsz = rows_left < group_m ? rows_left : group_m;
    const int32_t local = tile - g * per_group;
    TileCoord c;
    c.m_blk = first_m + local % gsz;
    c.n_blk = local / gsz;
    return c;
}

// Split-K over (tile, k-block) units for the skinny kernel: CTA c of G owns
// the contiguous unit range [unit_begin(c), unit_begin(c + 1)), where units
// are numbered tile-major (tile * k_blocks + kb).  Ranges differ in length by
// at most one unit.
TG_HD int64_t unit_begin(int64_t cta, int64_t num_ctas, int64_t total_units) {
    return (total_units * cta) / num_ctas;
}

// The CTA whose range holds unit u: the largest c with unit_begin(c) <= u,
// i.e. the largest c with total_units·c < (u + 1)·num_ctas.
TG_HD int64_t unit_owner(int64_t u, int64_t num_ctas, int64_t total_units) {
    return ((u + 1) * num_ctas + total_units - 1) / total_units - 1;
}

// The pair kernel's work items.  With T tiles on P clusters, W = T / P full
// waves are walked as above (cluster c takes tiles c, c + P, ...).  The
// R = T - W·P tiles of the last, partial wave may be shared out to otherwise
// idle clusters in one of two ways:
//  - H = 2 column halves: cluster c < 2R takes columns [128·(c % 2), +128)
//    of tail tile W·P + c / 2 over every k block, a 256×128 product that
//    needs no partial sums;
//  - S k-pieces: cluster c < R·S takes piece c % S (k blocks
//    [KB·j/S, KB·(j+1)/S) for j = c % S) of tile W·P + c / S; the pieces'
//    fp32 partials are summed in k order by whichever piece finishes last.
// S = H = 1 leaves the last wave whole.
constexpr int32_t kPairMaxSplit = 4;         // pieces per tail tile at most
constexpr int32_t kPairMinPieceBlocks = 8;   // k blocks per piece at least
// Choosing between the two, with times in 20ths of a whole tile's k block
// (fitted to interleaved timings of six shapes on GB300, K 4096 to 16384):
//  - a column half loads 1.5 times a whole tile's operand bytes per k block
//    for half its tensor work and runs a k block in about 17/20 of a whole
//    tile's time (both turn their operand rings over at about the same
//    bytes per cycle);
//  - S k-pieces run KB/S blocks each, then write and read back fp32 partial
//    sums, which costs about 7 + 4.5·S blocks' time.
// The cheapest of the two is taken; k-pieces need a workspace (KB = 0 rules
// them out).
constexpr int32_t kPairHalfBlockTime20 = 17;
constexpr int32_t kPairPieceCost20 = 140;     // fixed part of the partial-sum cost
constexpr int32_t kPairPieceCostPer20 = 90;   // and per piece

TG_HD int32_t pair_piece_time20(int32_t KB, int32_t S) {
    return 20 * KB / S + kPairPieceCost20 + kPairPieceCostPer20 * S;
}

// Clusters P to launch, k-pieces S and column halves H per tail tile, for T
// tiles of KB k blocks on at most `pairs` clusters.  At most one of S and H
// is above 1, and R·S·H <= P.
TG_HD void pair_launch_shape(int32_t T, int32_t pairs, int32_t KB, int32_t* P, int32_t* S,
                             int32_t* H) {
    const int32_t R = T >= pairs ? T % pairs : T;
    int32_t s = 1, h = 1;
    if (R > 0) {
        const int32_t fit = pairs / R;  // clusters per tail tile that are otherwise idle
        int32_t kmax = fit < kPairMaxSplit ? fit : kPairMaxSplit;
        if (kmax > KB / kPairMinPieceBlocks) kmax = KB / kPairMinPieceBlocks;
        int32_t best = fit >= 2 ? kPairHalfBlockTime20 * KB : 20 * KB;  // halves, or uncut
        for (int32_t k = 2; k <= kmax; ++k) {
            const int32_t t = pair_piece_time20(KB, k);
            if (t < best) {
                best = t;
                s = k;
            }
        }
        if (s == 1 && fit >= 2) h = 2;
    }
    *S = s;
    *H = h;
    const int32_t items = T * s * h;
    *P = T >= pairs ? pairs : (items < pairs ? items : pairs);
}

// Number of work items of cluster c.
TG_HD int32_t pair_item_count(int32_t c, int32_t T, int32_t P, int32_t S, int32_t H) {
    const int32_t W = T / P;
    const int32_t R = T - W * P;
    return W + (c < R * S * H ? 1 : 0);
}

// Item i of cluster c: its tile, k-block range [kb0, kb1) and column half
// (-1: all 256 columns; 0 or 1: columns [128·half, 128·half + 128)).
TG_HD void pair_item(int32_t c, int32_t i, int32_t T, int32_t P, int32_t S, int32_t H,
                     int32_t KB, int32_t* tile, int32_t* kb0, int32_t* kb1, int32_t* half) {
    const int32_t W = T / P;
    *half = -1;
    if (i < W) {
        *tile = c + i * P;
        *kb0 = 0;
        *kb1 = KB;
    } else if (H > 1) {
        *tile = W * P + c / H;
        *kb0 = 0;
        *kb1 = KB;
        *half = c % H;
    } else {
        const int32_t j = c % S;
        *tile = W * P + c / S;
        *kb0 = KB * j / S;
        *kb1 = KB * (j + 1) / S;
    }
}

}  // namespace tg
