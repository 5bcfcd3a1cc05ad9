// Persistent tile scheduler: the host-side partition of the mutable output
// into disjoint tiles ("cuTile Rust explained", "Ownership crosses the launch
// boundary": each tile program receives an exclusive output sub-tensor), turned
// into a static schedule for a persistent grid.
//
// CTA c of a grid of G CTAs owns the tiles with linear index t = c, c + G,
// c + 2G, ... < mt * nt. Each linear index maps to exactly one (m_tile,
// n_tile) pair, and each pair to exactly one index, so every output tile has
// exactly one owner and no two CTAs ever write the same element.
//
// The map is a grouped raster: the output is cut into bands of `group_m` tile
// rows; inside a band the index runs down the band's rows first and then
// across the columns. Tiles that run at the same time then share a few B
// column panels and A row panels, which keeps the operands of concurrently
// running tiles resident in L2.
#pragma once

#include <stdint.h>

namespace tpg {

struct TileCoord {
    int32_t m;
    int32_t n;
};

__host__ __device__ __forceinline__ TileCoord tile_of_index(int64_t t, int64_t mt, int64_t nt,
                                                          int32_t group_m) {
    const int64_t per_group = static_cast<int64_t>(group_m) * nt;
    const int64_t group = t / per_group;
    const int64_t first_m = group * group_m;
    const int64_t rows_here = (mt - first_m) < group_m ? (mt - first_m) : group_m;
    const int64_t local = t - group * per_group;
    TileCoord c;
    c.m = static_cast<int32_t>(first_m + local % rows_here);
    c.n = static_cast<int32_t>(local / rows_here);
    return c;
}

} // namespace tpg
