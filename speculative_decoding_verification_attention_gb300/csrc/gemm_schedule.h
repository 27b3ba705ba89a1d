// Work decompositions of the verify GEMM, shared by the kernels' roles (TMA
// producer, MMA issuer, epilogue) and by the host planner that the CPU tests
// enumerate.
//
// Weight streaming (M <= 256): stream-K.  Output tile t covers the 128 w
// rows (output columns) t * 128 ...  The first dp_tiles tiles are
// whole-tile work (CTA c takes c, c + G, c + 2G, ...); the k-block
// iterations of the remaining tiles are cut into G equal contiguous ranges,
// one per CTA, so every SM gets the same number of MMAs whatever the tile
// count.  The pieces of a tile cut between CTAs are added, in k order, by
// whichever piece is finished last.
//
// CTA pairs (M > 256): whole tiles of 256 rows and a ragged width.  The N
// columns are cut, in 32-column units, into tiles_n tiles whose widths
// differ by at most 32 (the first r tiles are 32 wider), so that
// tiles_m * tiles_n tiles spread evenly over the pairs; pair c takes tiles
// c, c + pairs, ...  Tile t covers rows (t % tiles_m) * 256 and the columns
// of N-tile t / tiles_m.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define SPEC_HD __host__ __device__ __forceinline__
#else
#define SPEC_HD inline
#endif

namespace spec {

struct SkGrid {
    int tiles_m, tiles, kblocks, G, dp_tiles;
    long long sk_iters;   // (tiles - dp_tiles) * kblocks
    SPEC_HD long long begin(int c) const { return sk_iters * c / G; }
};

struct Seg {
    int t, kb0, kb1;
};

struct SegWalker {
    SkGrid g;
    int c, w;
    long long it, end;
    SPEC_HD SegWalker(const SkGrid &g_, int c_)
        : g(g_), c(c_), w(0), it(g_.begin(c_)), end(g_.begin(c_ + 1)) {}
    SPEC_HD bool next(Seg &s)
    {
        if (w * g.G < g.dp_tiles) {
            s.t = c + w * g.G;
            s.kb0 = 0;
            s.kb1 = g.kblocks;
            ++w;
            return true;
        }
        if (it >= end) return false;
        const long long t = it / g.kblocks;
        s.t = g.dp_tiles + static_cast<int>(t);
        s.kb0 = static_cast<int>(it - t * g.kblocks);
        const long long left = end - it;
        s.kb1 = left < g.kblocks - s.kb0 ? s.kb0 + static_cast<int>(left) : g.kblocks;
        it += s.kb1 - s.kb0;
        return true;
    }
    // whether a segment follows the one next() returned last
    SPEC_HD bool has_more() const { return w * g.G < g.dp_tiles || it < end; }
};

struct PairGrid {
    int tiles_m, tiles_n;   // row tiles of 256, column tiles
    int q, r;               // N-tile nt is 32 * (q + (nt < r)) columns wide
    int kblocks;            // K / 64
    int pairs;              // CTA pairs launched
    SPEC_HD int tiles() const { return tiles_m * tiles_n; }
    SPEC_HD int width(int nt) const { return 32 * (q + (nt < r ? 1 : 0)); }
    SPEC_HD int col0(int nt) const { return 32 * (nt * q + (nt < r ? nt : r)); }
};

// For a segment that starts its tile (kb0 == 0) on unit c: the last unit
// holding a later piece of the same tile (c itself when the tile is whole).
// The pieces' holders are exactly units c+1 .. last.
SPEC_HD int sk_last_contributor(const SkGrid &g, int c, const Seg &s)
{
    int last = c;
    if (s.kb1 < g.kblocks) {
        const long long tile_end = static_cast<long long>(s.t - g.dp_tiles + 1) * g.kblocks;
        while (last + 1 < g.G && g.begin(last + 1) < tile_end) ++last;
    }
    return last;
}

// The unit whose stream-K range holds iteration x (0 <= x < sk_iters).
SPEC_HD int sk_unit_of(const SkGrid &g, long long x)
{
    int u = static_cast<int>(x * g.G / g.sk_iters);
    while (u + 1 < g.G && g.begin(u + 1) <= x) ++u;
    while (u > 0 && g.begin(u) > x) --u;
    return u;
}

// The units holding pieces of stream-K tile t (t >= dp_tiles): f .. l, in
// k order; f holds the first k-block.
SPEC_HD void sk_tile_units(const SkGrid &g, int t, int &f, int &l)
{
    const long long x0 = static_cast<long long>(t - g.dp_tiles) * g.kblocks;
    f = sk_unit_of(g, x0);
    l = sk_unit_of(g, x0 + g.kblocks - 1);
}

// Whether segment s of unit u is the first segment of u's stream-K range
// (a unit has at most two cut pieces: its first and its last segment).
SPEC_HD bool sk_first_segment(const SkGrid &g, int u, const Seg &s)
{
    return s.t >= g.dp_tiles &&
           static_cast<long long>(s.t - g.dp_tiles) * g.kblocks + s.kb0 == g.begin(u);
}

}  // namespace spec
