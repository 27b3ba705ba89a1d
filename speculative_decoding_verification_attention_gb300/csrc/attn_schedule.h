// Split of the verify-attention KV stream across CTA groups (host and
// device share this code).
//
// Unit = (sequence b, KV head h).  Unit (b, h) owns nk(b) = ceil(L_b / 128)
// key tiles; units are concatenated in (b, h) order into one stream of T
// tiles.  Group g processes the contiguous range [T*g/n, T*(g+1)/n) of that
// stream, so every group does the same number of tile steps whatever the
// mix of sequence lengths.  A range cut inside a unit yields a partial
// segment: group g writes the first such segment of its range to slot 2g
// and the last to slot 2g+1; a unit covered by one segment is written
// straight to the output.  The group whose range holds a split unit's last
// tile merges that unit's partials.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define SPEC_HD __host__ __device__ __forceinline__
#else
#define SPEC_HD inline
#endif

namespace spec {

constexpr int kKeyTile = 128;       // keys per tile
constexpr int kMinTilesPerGroup = 4;

// Tiles of sequence b, or 0 when kv_len is outside [1 + D, max_len].
SPEC_HD int seq_tiles(int32_t L, int D, int64_t max_len)
{
    return (L >= 1 + D && static_cast<int64_t>(L) <= max_len) ? (L + kKeyTile - 1) / kKeyTile : 0;
}

SPEC_HD int effective_groups(int64_t total, int groups)
{
    int64_t want = (total + kMinTilesPerGroup - 1) / kMinTilesPerGroup;
    if (want < 1) want = 1;
    return want < groups ? static_cast<int>(want) : groups;
}

SPEC_HD int64_t group_begin(int64_t total, int groups, int g)
{
    return total * g / groups;
}

// Largest g with group_begin(g) <= x (the group whose range holds x).
SPEC_HD int group_of(int64_t x, int64_t total, int groups)
{
    int64_t g = ((x + 1) * groups + total - 1) / total - 1;
    return g < groups - 1 ? static_cast<int>(g) : groups - 1;
}

struct Segment {
    int b, h;
    int tile_begin, tile_end;   // within the unit
    int slot;                   // -1: whole unit, written to the output
    int64_t unit_begin;         // stream position of the unit's first tile
    int nk;                     // tiles of the unit
};

// Walks the segments of one group's range.
struct SegmentWalker {
    const int32_t *kv_len;
    int B, D, Hkv;
    int64_t max_len;
    int g;
    int64_t gbegin, gend;
    // cursor
    int b, h, nk;
    int64_t unit_begin, pos;

    // Position the cursor at the unit holding stream position gbegin, given
    // the unit (b0, h0) and its first stream position.
    SPEC_HD void init(const int32_t *kv, int B_, int D_, int Hkv_, int64_t max_len_, int g_,
                      int64_t gb, int64_t ge, int b0, int h0, int64_t ub0)
    {
        kv_len = kv; B = B_; D = D_; Hkv = Hkv_; max_len = max_len_; g = g_;
        gbegin = gb; gend = ge;
        b = b0; h = h0; unit_begin = ub0; pos = gb;
        nk = (b < B) ? seq_tiles(kv_len[b], D, max_len) : 0;
    }

    SPEC_HD bool next(Segment &s)
    {
        if (pos >= gend) return false;
        while (nk == 0 || pos >= unit_begin + nk) {   // skip exhausted / empty units
            unit_begin += nk;
            if (++h == Hkv) { h = 0; ++b; }
            if (b >= B) return false;
            nk = seq_tiles(kv_len[b], D, max_len);
        }
        const int64_t end = gend < unit_begin + nk ? gend : unit_begin + nk;
        s.b = b; s.h = h; s.nk = nk; s.unit_begin = unit_begin;
        s.tile_begin = static_cast<int>(pos - unit_begin);
        s.tile_end = static_cast<int>(end - unit_begin);
        if (s.tile_begin == 0 && s.tile_end == nk) s.slot = -1;
        else s.slot = (unit_begin <= gbegin) ? 2 * g : 2 * g + 1;
        pos = end;
        return true;
    }
};

// Serial locate of stream position x: returns (b, h, unit_begin) of the unit
// holding x and the total tile count (host reference; the kernels use a
// block-parallel version of the same scan).
SPEC_HD int64_t total_tiles_serial(const int32_t *kv, int B, int D, int Hkv, int64_t max_len)
{
    int64_t t = 0;
    for (int b = 0; b < B; ++b) t += static_cast<int64_t>(Hkv) * seq_tiles(kv[b], D, max_len);
    return t;
}

SPEC_HD void locate_serial(const int32_t *kv, int B, int D, int Hkv, int64_t max_len, int64_t x,
                           int &b_out, int &h_out, int64_t &ub_out)
{
    int64_t acc = 0;
    for (int b = 0; b < B; ++b) {
        const int nk = seq_tiles(kv[b], D, max_len);
        const int64_t span = static_cast<int64_t>(Hkv) * nk;
        if (nk > 0 && x < acc + span) {
            const int h = static_cast<int>((x - acc) / nk);
            b_out = b; h_out = h; ub_out = acc + static_cast<int64_t>(h) * nk;
            return;
        }
        acc += span;
    }
    b_out = B; h_out = 0; ub_out = acc;
}

}  // namespace spec
