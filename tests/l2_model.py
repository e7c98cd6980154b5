"""An LRU model of L2 for the persistent kernel's whole-tile order.

Every cluster runs its tiles round-robin (tile c, c + G, ...) in the raster
order, and all clusters advance one k-block at a time, reading the A slab of
their tile's row strip and the B slab of its column strip (256 rows × 64 k,
32 KiB each).  The model replays that access order through a least-recently
used cache of `capacity` bytes and counts the bytes it misses.  With 63 MB of
capacity it reproduces the measured DRAM reads of the up-only k order at
8192³ for raster group widths 2 to 32 (1.79, 1.28, 1.09, 1.31, 2.06 GB
modelled against 1.92, 1.34, 1.05, 1.25, 2.10 GB measured), which is what
the plan's k-order rule (alternate the k direction of odd waves above 60 MB
of strips a wave) rests on.
"""
from collections import OrderedDict

SLAB = 256 * 64 * 2   # bytes of one strip's k-block slab


def raster(m_tiles, n_tiles, swizzle):
    """The kernel's tile raster: groups of `swizzle` tile columns, rows in
    order inside a group, odd groups taking their rows in reverse."""
    order = []
    for g, n0 in enumerate(range(0, n_tiles, swizzle)):
        w = min(swizzle, n_tiles - n0)
        rows = range(m_tiles - 1, -1, -1) if g % 2 else range(m_tiles)
        for m in rows:
            for j in range(w):
                order.append((m, n0 + j))
    return order


def dram_bytes(m_tiles, n_tiles, k_blocks, clusters, swizzle=8, alternate=False, capacity=63_000_000):
    """Modelled DRAM bytes read by one launch of whole tiles."""
    order = raster(m_tiles, n_tiles, swizzle)
    cap = capacity // SLAB
    cache = OrderedDict()
    misses = 0
    for w0 in range(0, len(order), clusters):
        wave = order[w0:w0 + clusters]
        down = alternate and (w0 // clusters) % 2 == 1
        for kb in (range(k_blocks - 1, -1, -1) if down else range(k_blocks)):
            for (m, n) in wave:
                for key in (("A", m, kb), ("B", n, kb)):
                    if key in cache:
                        cache.move_to_end(key)
                    else:
                        misses += 1
                        cache[key] = None
                        if len(cache) > cap:
                            cache.popitem(last=False)
    return misses * SLAB
