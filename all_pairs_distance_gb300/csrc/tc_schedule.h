// Work-unit schedule of the tensor-core sweeps (host and device).
//
// Pure integer functions, kept apart from the kernel so that a host program
// can enumerate the units and check that they cover every tile pair once.
#pragma once

#ifndef __CUDACC__
#include <algorithm>
#define TC_HD inline
using std::max;
using std::min;
#else
#define TC_HD __host__ __device__ __forceinline__
#endif

namespace dbscan {

// Units go column chunk by column chunk (TC_CHUNK tiles each), and within a
// chunk by row unit: the CTAs working at the same time stream the same chunk of
// column tiles, which stays in L2 even when the operand arrays do not.  A row
// unit is rt consecutive row blocks rb .. rb + rt - 1 (rb = rt x its index);
// every column tile staged for it meets all of them, so a column tile is
// copied from L2 once per rt row blocks.  A unit is a row unit against the
// chunk's tiles t with t - rb in [lo, hi) (the whole triangle for the count,
// a distance band for the union, every tile for the border's rectangle).  In
// the triangle the pairs (rb + r, t) with t < rb + r are skipped; every pair
// (r, t) with t >= r still lies in exactly one unit and one band, since bands
// split t - rb.  (The union's bands start at distance 1 and it skips the pair
// (rb + 1, rb + 1) too: diagonal tiles are joined by the tile-local union.)
// Union bands: tile distances [edge_b, edge_{b+1}) from the diagonal (-1 = no
// upper limit), nearest first.  The diagonal itself (distance 0) is left out:
// the tile-local union has already joined every neighbour pair inside a tile.
// Three bands measured faster than six (1M x 3 union 1.55 -> 1.29 ms,
// 100k x 2 0.54 -> 0.43 ms, 500k x 64 2.71 -> 2.48 ms): every band costs a
// compression, a tile-root snapshot and the sweep's fixed start-up.
constexpr int UNION_BANDS = 3;
constexpr int kUnionBandEdges[UNION_BANDS + 1] = {1, 4, 16, -1};

constexpr int TC_CHUNK = 512;
// The union's last band (no upper distance) over at most 2,048 column tiles
// takes chunks of 128: the box test keeps few of its tiles, scattered, and a
// long chunk can leave one unit with hundreds of kept tiles at the end of the
// sweep (200k x 16: 588 tile pairs in one unit against 12 on average; union
// 0.91 -> 0.77 ms).  With more tiles the units' own box scans outweigh that
// (1M x 3: 1.37 -> 2.17 ms with short chunks).
constexpr int TC_FAR_CHUNK = 128;
constexpr int TC_FAR_CHUNK_MAX_TILES = 2048;
constexpr int TC_TILE = 128;   // points per tile (BT)
TC_HD int tc_chunk(int union_band, int hi, int n_cols) {
    const int nct = (n_cols + TC_TILE - 1) / TC_TILE;
    return union_band && hi < 0 && nct <= TC_FAR_CHUNK_MAX_TILES ? TC_FAR_CHUNK : TC_CHUNK;
}
struct TcSched {
    int nrt, nct, nchunks, rt, nru, chunk;
    unsigned units;
};
// The row units [first, first + count) of chunk c that have at least one tile
// in it: rb + lo < (c + 1) * chunk and, with an upper distance,
// rb + hi > c * chunk.
TC_HD int chunk_first_row(const TcSched &s, int c, int tri, int hi) {
    if (!(tri && hi >= 0)) return 0;
    const int x = c * s.chunk - hi;          // first rb with rb > x
    return x < 0 ? 0 : x / s.rt + 1;
}
TC_HD int chunk_rows(const TcSched &s, int c, int tri, int lo, int hi) {
    if (!tri) return s.nru;
    const int lim = (c + 1) * s.chunk - lo;  // rb < lim
    const int end = lim <= 0 ? 0 : min(s.nru, (lim + s.rt - 1) / s.rt);
    return max(0, end - chunk_first_row(s, c, tri, hi));
}
TC_HD TcSched tc_sched(int n_rows, int n_cols, int tri, int lo, int hi, int rt, int chunk) {
    TcSched s;
    s.nrt = (n_rows + TC_TILE - 1) / TC_TILE;
    s.nct = (n_cols + TC_TILE - 1) / TC_TILE;
    s.chunk = chunk;
    s.nchunks = (s.nct + chunk - 1) / chunk;
    s.rt = rt;
    s.nru = (s.nrt + rt - 1) / rt;
    long long u = 0;
    for (int c = 0; c < s.nchunks; ++c) u += chunk_rows(s, c, tri, lo, hi);
    s.units = (unsigned)u;
    return s;
}
// Unit u -> first row block, row blocks in the unit and column tiles [t0, t1);
// false when it holds none.
TC_HD bool tc_unit(const TcSched &s, unsigned u, int tri, int lo, int hi, int &rb, int &nrow,
                   int &t0, int &t1) {
    int c = 0;
    for (; c < s.nchunks; ++c) {
        const unsigned r = (unsigned)chunk_rows(s, c, tri, lo, hi);
        if (u < r) break;
        u -= r;
    }
    rb = (chunk_first_row(s, c, tri, hi) + (int)u) * s.rt;
    nrow = min(s.rt, s.nrt - rb);
    t0 = max(c * s.chunk, tri ? rb + lo : 0);
    t1 = min(min((c + 1) * s.chunk, s.nct), (tri && hi >= 0) ? rb + hi : s.nct);
    return t0 < t1;
}

}  // namespace dbscan
