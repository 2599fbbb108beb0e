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

}  // namespace tg
