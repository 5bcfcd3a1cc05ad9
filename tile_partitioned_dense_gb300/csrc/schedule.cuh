// Persistent tile scheduler: the host-side partition of the mutable output
// into disjoint tiles ("cuTile Rust explained", "Ownership crosses the launch
// boundary": each tile program receives an exclusive output sub-tensor), turned
// into a static schedule for a persistent grid.
//
// The output is a grid of mt x nt tiles (rows of BM, columns of BN). A grid of
// P workers (CTAs, or CTA pairs) walks a single linear index t = w, w + P,
// w + 2P, ... for worker w:
//   - indices t < whole are whole tiles, mapped to (m, n) by a grouped raster;
//   - indices whole <= t < whole + pieces are column pieces of the remaining
//     tiles: tile whole + (t - whole) / split, piece (t - whole) % split, each
//     BN / split columns wide.
// whole is a multiple of P (the complete rounds), so the pieces start a new
// round. Cutting a nearly empty last round (or, with fewer tiles than workers,
// every tile) into column pieces lets more workers share it instead of leaving
// most of them idle while some finish a whole tile (wave quantization). Every
// (tile, piece) pair has exactly one index, so every output element has
// exactly one owner: no atomics, no split-K.
//
// The grouped raster: the tile grid is cut into bands of `group_m` tile rows;
// inside a band the index runs down the band's rows first, then across the
// columns, so tiles that run at the same time share a few B column panels and
// A row panels and keep them resident in L2.
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

struct Schedule {
    int64_t mt, nt;  // tile grid
    int32_t group_m; // band height of the grouped raster, in tiles
    int32_t split;   // 1, 2 or 4: column pieces per tile after the whole rounds
    int64_t whole;   // tiles processed whole (a multiple of the worker count)
    int64_t pieces;  // split * (mt * nt - whole)
    int64_t workers; // persistent workers to launch
};

// One unit of work: tile row m (in tiles), first column n and width (in columns).
struct WorkItem {
    int32_t m;
    int32_t n;
    int32_t width;
};

// The unit with linear index t, or false past the end.
__host__ __device__ __forceinline__ bool work_item(const Schedule &s, int64_t t, int32_t bn,
                                                   WorkItem &w) {
    if (t < s.whole) {
        const TileCoord c = tile_of_index(t, s.mt, s.nt, s.group_m);
        w.m = c.m;
        w.n = c.n * bn;
        w.width = bn;
        return true;
    }
    const int64_t u = t - s.whole;
    if (u >= s.pieces) return false;
    const TileCoord c = tile_of_index(s.whole + u / s.split, s.mt, s.nt, s.group_m);
    const int32_t width = bn / s.split;
    w.m = c.m;
    w.n = c.n * bn + static_cast<int32_t>(u % s.split) * width;
    w.width = width;
    return true;
}

// Host-side choice for at most `cap` persistent workers. With at least `cap`
// tiles: whole rounds of whole tiles, then the remaining tiles cut into
// `split` column pieces; with fewer tiles than workers every tile is cut, so
// that more workers have work. split is taken from {1, 2, 4} (up to
// max_split) to minimise the estimated time of the cut part: its rounds times
// the cost of one piece. A piece 1/f of a tile wide still loads all of the
// tile's A rows, so it is costed at a_share + (1 - a_share) / f of a whole
// tile, a_share being A's part of the operand bytes a whole tile loads per
// k-block. With max_split = 2 the choice is the same for any piece cost
// between 1/2 and 1 of a tile: halves win exactly when 2 * rest <= cap.
__host__ __device__ __forceinline__ Schedule make_schedule(int64_t mt, int64_t nt, int32_t group_m, int64_t cap,
                                                           int32_t max_split, double a_share) {
    Schedule s;
    s.mt = mt;
    s.nt = nt;
    s.group_m = group_m;
    const int64_t total = mt * nt;
    if (cap < 1) cap = 1;
    const int64_t rest = total >= cap ? total - (total / cap) * cap : total;
    int32_t best = 1;
    double best_cost = 1e300;
    for (int32_t f = 1; f <= max_split && f <= 4; f *= 2) {
        const double rounds = static_cast<double>((f * rest + cap - 1) / cap);
        const double cost = rounds * (a_share + (1.0 - a_share) / f);
        if (cost < best_cost - 1e-9) {
            best_cost = cost;
            best = f;
        }
    }
    s.split = best;
    if (total >= cap) {
        s.workers = cap;
        s.whole = (total / cap) * cap;
        s.pieces = s.split * (total - s.whole);
    } else {
        s.whole = 0;
        s.pieces = s.split * total;
        s.workers = s.pieces < cap ? s.pieces : cap;
        if (s.workers < 1) s.workers = 1;
    }
    return s;
}

} // namespace tpg
