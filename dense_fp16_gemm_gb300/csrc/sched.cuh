// Tile scheduling shared by the kernel and the host: the swizzled raster and the
// multiply-shift division it uses.  Everything here is plain integer code that
// compiles for both sides, so the host tests exercise the exact function the
// kernel runs.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define G16_HD __host__ __device__ __forceinline__
#else
#define G16_HD inline
#endif

namespace g16 {

// Division by a divisor that is fixed for a whole launch but unknown at compile
// time, as one multiply-high, one add and one shift (Granlund & Montgomery,
// "Division by Invariant Integers using Multiplication", PLDI 1994, the
// round-up method of their Figure 4.1).  With l = ceil(log2 d) and
// mul = floor(2^32 (2^l - d) / d) + 1, q = (mulhi(mul, n) + n) >> l for every
// 0 <= n < 2^31 (the sum then fits in 32 bits).  Requires 1 <= d <= 2^31.
struct FastDiv {
    uint32_t d;
    uint32_t mul;
    uint32_t shift;
};

G16_HD FastDiv make_fastdiv(uint32_t d) {
    FastDiv f;
    f.d = d;
    uint32_t l = 0;
    while (l < 31 && (uint64_t(1) << l) < d) ++l;
    f.shift = l;
    f.mul = uint32_t((((uint64_t(1) << l) - d) << 32) / d + 1);
    return f;
}

G16_HD uint32_t fastdiv_q(const FastDiv& f, uint32_t n) {
#if defined(__CUDA_ARCH__)
    uint32_t hi = __umulhi(n, f.mul);
#else
    uint32_t hi = uint32_t((uint64_t(n) * f.mul) >> 32);
#endif
    return (hi + n) >> f.shift;
}

// The tile raster.  Output tiles form an m_tiles × n_tiles grid.  The N axis is
// cut into groups of `swizzle` tile columns (the last group holds what is
// left); a linear index walks the groups in order and, inside a group, goes
// row-major (n fastest).  Consecutive indices, which run at the same time in a
// persistent grid, therefore share a few B column strips and a few A row
// strips, and those stay in L2.  Tilus matmul-hopper tutorial, "4. Pipeline
// Abstraction and Two Consumer Warp Groups", §Tile Rasterization (the mapping
// and its narrower last group).  One change to it: odd groups take their rows
// in reverse (a serpentine), so that a group starts on the A row strips the
// previous group's last wave has just read, instead of on rows read long ago.
struct Raster {
    uint32_t m_tiles;
    uint32_t n_tiles;
    uint32_t swizzle;
    FastDiv group;  // tiles per full group: m_tiles * swizzle
    FastDiv full;   // width of a full group
    FastDiv last;   // width of the last group
};

G16_HD Raster make_raster(uint32_t m_tiles, uint32_t n_tiles, uint32_t swizzle) {
    Raster r;
    if (swizzle > n_tiles) swizzle = n_tiles;
    if (swizzle < 1) swizzle = 1;
    r.m_tiles = m_tiles;
    r.n_tiles = n_tiles;
    r.swizzle = swizzle;
    uint32_t rem = n_tiles % swizzle;
    r.group = make_fastdiv(m_tiles * swizzle);
    r.full = make_fastdiv(swizzle);
    r.last = make_fastdiv(rem ? rem : swizzle);
    return r;
}

// linear index t in [0, m_tiles*n_tiles) -> (m_tile, n_tile)
G16_HD void raster_coord(const Raster& r, uint32_t t, uint32_t& m_tile, uint32_t& n_tile) {
    uint32_t g = fastdiv_q(r.group, t);
    uint32_t in = t - g * r.group.d;
    uint32_t first_n = g * r.swizzle;
    const FastDiv& w = (first_n + r.swizzle <= r.n_tiles) ? r.full : r.last;
    uint32_t mm = fastdiv_q(w, in);
    m_tile = (g & 1u) ? r.m_tiles - 1u - mm : mm;
    n_tile = first_n + (in - mm * w.d);
}

// Kinds of work item (see work_next)
enum : uint32_t { kItemWhole = 0, kItemPartialOut = 1, kItemOwner = 2, kItemSplitPiece = 3 };

// ---------------------------------------------------------------------------
// work schedule
// ---------------------------------------------------------------------------
// The functions below take the launch's parameters as any struct P with the
// fields num_tiles, num_kb, sk_tiles, sk_units, tail_first, tail_split and
// split_pieces, so
// that the host tests enumerate exactly the items the kernel runs.
//
// The tiles [0, sk_tiles) form the stream-K part: their sk_tiles * num_kb
// k-block units are split into G equal contiguous ranges, one per cluster, so
// the last, partly filled wave of a purely tile-parallel schedule is spread
// over every cluster.  The rest of the tiles go round-robin, whole.  A range
// may start or end inside a tile:
//   - a piece that does not start at k-block 0 (only ever a cluster's first
//     item) is written as an fp32 partial tile to the cluster's workspace slot
//     and published with a release flag; its k-blocks run from the last one
//     down, so that all clusters' first pieces end at the same k-block;
//   - the piece that starts at k-block 0 but stops early is the tile's owner:
//     it waits for the partials of the clusters that took the rest of the tile
//     (the next ones in order), adds them in that order and stores C.
// Owner pieces come at the end of a cluster's range and partial pieces at the
// start, so an owner seldom waits.
//
// Split pieces (split_pieces = s > 1, only when every cluster runs exactly one
// item): tile c / s is cut along k into s pieces of equal length, piece c % s
// on cluster c.  The pieces of a tile are symmetric: the tile's columns are cut
// into s contiguous slices, piece i owning slice i; each piece writes the fp32
// partial of the slices it does not own, publishes a flag, waits for the other
// pieces' flags, and reduces its own slice, adding the s partials in piece
// order, which is k order.  So the fix-up is spread over all s clusters
// instead of falling on one owner.
//
// After the whole tiles come the N-split items: the last tiles of the raster,
// [tail_first, num_tiles), each cut into tail_split column slices of
// BN/tail_split, dealt round-robin like the whole tiles.  No cluster depends
// on another's result.  A slice's main loop is nearly as long as a whole tile's
// (a narrower MMA is not proportionally faster); its epilogue drains
// 1/tail_split of the accumulator.

struct Item {
    uint32_t tile;
    uint32_t kb0, kb1;   // k-block range [kb0, kb1)
    uint32_t kind;
    uint32_t part, parts;   // column slice `part` of `parts` (1 = the whole tile)
    uint32_t piece, pieces; // split piece `piece` of `pieces` (1 = not split)
};

struct Work {
    uint64_t u, u_end;   // this cluster's stream-K units still to do
    uint32_t t;          // next whole tile
    uint32_t q;          // next N-split tail item
    uint32_t G;          // clusters
    uint32_t c;          // this cluster
    uint32_t claimed;    // 1 once this cluster has asked for a last-wave tile
};

template <class P>
G16_HD uint64_t sk_begin(const P& p, uint32_t c, uint32_t G) {
    return p.sk_units * c / G;
}

template <class P>
G16_HD void work_init(Work& s, const P& p, uint32_t c, uint32_t G) {
    s.u = sk_begin(p, c, G);
    s.u_end = sk_begin(p, c + 1, G);
    s.t = p.sk_tiles + c;
    s.q = c;
    s.G = G;
    s.c = c;
    s.claimed = 0;
    if (p.split_pieces > 1) {   // one split piece per cluster, nothing else
        s.u = s.u_end = 0;
        s.t = c;                 // reused: this cluster's piece index in the launch
        s.q = 1;                 // 1 while the piece is still to be returned
    }
}

// The next work item of a cluster.  Whole tiles in [dyn_first, num_tiles)
// (the last, partial wave) are not dealt round-robin: once a cluster has run
// its share, it asks `claim` for one, and gets a tile of that range or
// num_tiles (none left); the kernel's claim hands them to the clusters that
// finish first.
template <class P, class Claim>
G16_HD bool work_next(Work& s, const P& p, Item& it, Claim&& claim) {
    it.piece = 0;
    it.pieces = 1;
    if (p.split_pieces > 1) {
        if (!s.q) return false;
        s.q = 0;
        const uint32_t np = p.split_pieces, piece = s.t % np;
        it.tile = s.t / np;
        it.kb0 = uint32_t(uint64_t(p.num_kb) * piece / np);
        it.kb1 = uint32_t(uint64_t(p.num_kb) * (piece + 1) / np);
        it.kind = kItemSplitPiece;
        it.part = 0;
        it.parts = 1;
        it.piece = piece;
        it.pieces = np;
        return true;
    }
    if (s.u < s.u_end) {
        const uint32_t t = uint32_t(s.u / p.num_kb);
        const uint32_t kb0 = uint32_t(s.u - uint64_t(t) * p.num_kb);
        const uint64_t left = s.u_end - s.u;
        const uint32_t kb1 = left >= uint64_t(p.num_kb - kb0) ? p.num_kb : kb0 + uint32_t(left);
        it.tile = t;
        it.kb0 = kb0;
        it.kb1 = kb1;
        it.kind = kb0 > 0 ? kItemPartialOut : (kb1 < p.num_kb ? kItemOwner : kItemWhole);
        it.part = 0;
        it.parts = 1;
        s.u += kb1 - kb0;
        return true;
    }
    it.kb0 = 0;
    it.kb1 = p.num_kb;
    it.kind = kItemWhole;
    it.part = 0;
    it.parts = 1;
    if (s.t < p.tail_first && s.t < p.dyn_first) {
        it.tile = s.t;
        s.t += s.G;
        return true;
    }
    if (p.dyn_first < p.num_tiles) {   // (no N-split tail then)
        if (s.claimed) return false;
        s.claimed = 1;
        it.tile = claim();
        return it.tile < p.num_tiles;
    }
    if (s.q < (p.num_tiles - p.tail_first) * p.tail_split) {
        it.tile = p.tail_first + s.q / p.tail_split;
        it.part = s.q % p.tail_split;
        it.parts = p.tail_split;
        s.q += s.G;
        return true;
    }
    return false;
}

// The same, with the claims of the last wave modelled as taken in cluster
// order (cluster c gets the c-th tile of the range): one of the orders the
// kernel can produce, for host-side enumeration and tests.
template <class P>
G16_HD bool work_next(Work& s, const P& p, Item& it) {
    return work_next(s, p, it, [&]() -> uint32_t {
        const uint32_t t = p.dyn_first + s.c;
        return t < p.num_tiles ? t : p.num_tiles;
    });
}

// Whether the producer loads an item's k-blocks from the last one down.  A
// partial stream-K piece does (so that at a launch's start the pieces of all
// clusters read the same k-slab together).  A whole tile after the stream-K
// region does in odd rounds, round = (tile - sk_tiles) / G: all clusters
// stream k-blocks up in one round and down in the next, so a round begins on
// the k-slabs of the A and B strips that the round before read last, which
// are still in L2, instead of on those it read first, which a cache that
// holds less than a round's strips has evicted (only when the launch's plan
// says so, p.k_alternate: when one round's strips exceed the share of L2 that
// holds them).  It is a function of the tile and the launch alone, so the same
// tile takes the same k order in every schedule that runs it whole or in
// column slices.
template <class P>
G16_HD bool item_k_down(const P& p, const Item& it, uint32_t G) {
    if (it.kind == kItemPartialOut) return true;
    if (!p.k_alternate || it.kind != kItemWhole || it.tile < p.sk_tiles) return false;
    return (((it.tile - p.sk_tiles) / G) & 1u) != 0;
}

// The number of clusters after cluster c whose stream-K ranges start inside
// `tile`: the partners whose partial tiles the owner of `tile` (cluster c, the
// piece from k-block 0) adds, in cluster order, which is k order.
template <class P>
G16_HD uint32_t owner_partners(const P& p, uint32_t tile, uint32_t c, uint32_t G) {
    const uint64_t tile_end = uint64_t(tile + 1) * p.num_kb;
    uint32_t n = 0;
    while (c + 1 + n < G && sk_begin(p, c + 1 + n, G) < tile_end) ++n;
    return n;
}

// The schedule fields of a launch's parameters, from its plan.  PlanT is the
// library's plan struct; P any struct with the fields read above.
template <class P, class PlanT>
inline void set_schedule(P& p, const PlanT& pl) {
    p.num_tiles = uint32_t(pl.num_tiles);
    p.num_kb = uint32_t(pl.k_blocks);
    p.sk_tiles = uint32_t(pl.sk_tiles);
    p.sk_units = uint64_t(pl.sk_tiles) * uint64_t(pl.k_blocks);
    p.tail_split = uint32_t(pl.tail_split > 1 ? pl.tail_split : 1);
    p.tail_first = uint32_t(pl.num_tiles - (pl.tail_split > 1 ? pl.tail_tiles : 0));
    p.split_pieces = uint32_t(pl.split_pieces > 1 ? pl.split_pieces : 1);
    p.k_alternate = uint32_t(pl.k_order == 1 ? 1 : 0);
    p.dyn_first = uint32_t(pl.num_tiles - (pl.claimed_tiles > 0 ? pl.claimed_tiles : 0));
}

}  // namespace g16
