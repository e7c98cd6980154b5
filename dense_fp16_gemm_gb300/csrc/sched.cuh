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

}  // namespace g16
