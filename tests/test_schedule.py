"""The persistent schedule, enumerated on the host with the kernel's own code.

gemm_f16_nt_schedule runs the same work_init / work_next / owner_partners
functions the kernel runs (they are compiled for both sides), from the same
plan.  These tests check, for many shapes and options, what the kernel relies
on without checking it itself:
  - every (tile, column quarter, k-block) is computed exactly once;
  - a cluster has at most one partial piece, and it is its first item (the
    workspace holds one partial tile per cluster);
  - a tile's owner adds exactly the partial pieces of that tile, and they are
    held by the clusters right after it, in k order;
  - the stream-K ranges are balanced across clusters to one k-block;
  - the plan's N-split is what the clusters run;
  - each item's coordinates are the raster's.
Small problems default to the small-problem kernel, whose plan has one tile
per cluster (tile c at m_tile = c % m_tiles, n_tile = c / m_tiles, all of k);
the same checks cover it, and the cases that name cta_group 2 keep the
persistent kernel for those shapes.
"""
import pytest

import dense_fp16_gemm_gb300 as g

WHOLE, PARTIAL, OWNER, SPLIT = 0, 1, 2, 3

CASES = [
    # M, N, K, options, max_clusters
    (4096, 4096, 4096, {}, 76),                       # stream-K: last wave + one wave
    (6144, 4096, 4096, {}, 76),
    (4096, 11008, 4096, {}, 76),
    (8192, 8192, 8192, {}, 76),                       # whole tiles
    (8192, 8192, 8192, {"schedule": 2}, 76),          # stream-K forced
    (8192, 8192, 8192, {"schedule": 3}, 76),          # N-split tail forced
    (256, 256, 256, {}, 76),                          # small-problem kernel: 16 tiles of 128 x 32
    (256, 256, 256, {"cta_group": 2}, 76),            # persistent: N-split in four
    (256, 256, 8192, {"cta_group": 2}, 76),           # one tile cut in k
    (1024, 1024, 8192, {"cta_group": 2}, 64),         # 16 tiles cut in k
    (1024, 1024, 1024, {}, 76),                       # small-problem kernel: 128 tiles of 128 x 64
    (1024, 1024, 1024, {"cta_group": 2}, 76),
    (512, 4096, 4096, {}, 76),                        # small-problem kernel: 128 x 128 tiles
    (300, 520, 328, {"schedule": 5, "cta_group": 2, "tile_n": 64}, 76),   # forced: pairs, 256 x 64
    (4096, 4096, 1024, {}, 76),                       # shallow last wave: N-split
    (4000, 3000, 5000, {"_lib": "mcast"}, 36),        # two pairs per cluster (multicast build's default)
    (4000, 3000, 5000, {}, 76),                       # one pair: the default build
    (4000, 3000, 5000, {"schedule": 2, "cluster_pairs": 1}, 76),
    (300, 520, 328, {"schedule": 2}, 76),
    (1300, 1000, 320, {"schedule": 3, "cluster_pairs": 1}, 76),
    (700, 900, 1000, {"cta_group": 1}, 152),
    (700, 900, 1000, {"cta_group": 1, "schedule": 2}, 152),
    (1, 1, 1, {}, 76),
    (1, 1, 1, {"cta_group": 2}, 76),
    (70000, 300, 64, {}, 76),
    (256, 512, 1 << 20, {}, 76),
    (1024, 1024, 8192, {"cta_group": 2}, 76),         # split pieces: 16 tiles x 4
    (256, 256, 8192, {"cta_group": 2}, 76),           # one tile in 8 pieces
    (256, 256, 16384, {}, 76),                        # small-problem kernel, split-K: 16 tiles x 8 pieces
    (300, 200, 3000, {}, 76),                         # small-problem kernel, split-K: 21 tiles x 4 pieces
    (256, 256, 1 << 17, {}, 76),                      # too deep a piece: persistent split pieces
    (300, 520, 328, {"schedule": 4}, 76),             # forced: pieces of 1 or 2 k-blocks
    (700, 900, 1000, {"cta_group": 1, "schedule": 4}, 152),
]


def _random_cases(n=60, seed=20261203):
    """Seeded random problems and options, sizes log-uniform in 1..20000 (K up to 2^17)."""
    import numpy as np
    rng = np.random.default_rng(seed)
    size = lambda hi: int(np.clip(np.round(np.exp(rng.uniform(0.0, np.log(hi)))), 1, hi))
    out = []
    for _ in range(n):
        cg = 1 if rng.random() < 0.25 else 2
        opts = {"cta_group": cg, "schedule": int(rng.choice([0, 0, 1, 2, 3, 4]))}
        if cg == 2:
            opts["cluster_pairs"] = int(rng.choice([0, 1, 2]))
        mc = int(rng.choice([0, 0, 7, 36, 64, 76, 152]))
        out.append((size(20000), size(20000), size(1 << 17), opts, mc))
    return out


CASES = CASES + _random_cases()


def _all_items(M, N, K, opts, max_clusters):
    """The plan and every cluster's items.  Two pairs per cluster exist only in
    the multicast build, whose schedule code is the same source; it is asked
    for them explicitly (cluster_pairs 2) or by "_lib"."""
    opts = dict(opts)
    lib = opts.pop("_lib", None)
    lib = g.library_mcast() if (lib == "mcast" or opts.get("cluster_pairs") == 2) else g.library()
    o = g.Options(**opts)
    pl = g.plan(M, N, K, max_clusters=max_clusters, options=o, lib=lib)
    items = [g.schedule(M, N, K, c, max_clusters=max_clusters, options=o, lib=lib)
             for c in range(pl["clusters"])]
    return pl, items


def check_coverage(pl, items):
    """Every (tile, column quarter, k-block) exactly once; the plan's N-split realized."""
    kb = pl["k_blocks"]
    seen = {}
    sliced = 0
    for c, its in enumerate(items):
        for it in its:
            assert it["parts"] in (1, pl["tail_split"]), it
            # (the persistent kernel's split pieces; the small kernel's split-K uses owners)
            assert (it["kind"] == SPLIT) == (pl["split_pieces"] > 1 and pl["kernel"] == 0), it
            if it["parts"] > 1:
                sliced += 1
                assert it["tile"] >= pl["num_tiles"] - pl["tail_tiles"], it
            q = 4 // it["parts"]
            for quarter in range(it["part"] * q, (it["part"] + 1) * q):
                for k in range(it["kb0"], it["kb1"]):
                    key = (it["tile"], quarter, k)
                    assert key not in seen, (key, c, seen.get(key))
                    seen[key] = c
    assert len(seen) == pl["num_tiles"] * 4 * kb
    assert sliced == (pl["tail_tiles"] * pl["tail_split"] if pl["tail_split"] > 1 else 0)


def check_split_pieces(pl, items):
    """Split pieces: each cluster runs exactly one piece; cluster c holds piece
    c % s of tile c // s; a tile's pieces cover its k-blocks in order, with
    lengths differing by at most one."""
    s, kb = pl["split_pieces"], pl["k_blocks"]
    assert pl["clusters"] == pl["num_tiles"] * s and pl["sk_tiles"] == 0 and pl["tail_split"] == 1
    for c, its in enumerate(items):
        assert len(its) == 1, (c, its)
        it = its[0]
        assert (it["kind"], it["tile"], it["piece"], it["pieces"], it["parts"]) == (SPLIT, c // s, c % s, s, 1)
        assert it["kb0"] == kb * (c % s) // s and it["kb1"] == kb * (c % s + 1) // s
    lens = [its[0]["kb1"] - its[0]["kb0"] for its in items]
    assert max(lens) - min(lens) <= 1 and min(lens) >= 1


def check_partials_and_owners(pl, items):
    """One partial piece per cluster at most, as its first item; owners add exactly
    the partial pieces of their tile, held by the next clusters, contiguous in k."""
    if pl["split_pieces"] > 1 and pl["kernel"] == 0:
        check_split_pieces(pl, items)
        return
    kb = pl["k_blocks"]
    # tiles that may be split in k: the stream-K tiles, or (small-problem kernel
    # with split-K) every tile
    split_tiles = pl["num_tiles"] if pl["kernel"] == 1 and pl["split_pieces"] > 1 else pl["sk_tiles"]
    partial_of = {}                                   # tile -> [(cluster, kb0, kb1)]
    for c, its in enumerate(items):
        partials = [i for i, it in enumerate(its) if it["kind"] == PARTIAL]
        assert partials in ([], [0]), (c, its)        # one workspace slot per cluster
        for it in its:
            if it["kind"] != WHOLE:
                assert it["parts"] == 1 and it["tile"] < split_tiles
            if it["kind"] == PARTIAL:
                assert 0 < it["kb0"] < it["kb1"] <= kb     # a middle piece ends inside the tile
                partial_of.setdefault(it["tile"], []).append((c, it["kb0"], it["kb1"]))
            elif it["kind"] == OWNER:
                assert it["kb0"] == 0 < it["kb1"] < kb
            else:
                assert (it["kb0"], it["kb1"]) == (0, kb) and it["partners"] == 0
    owners = 0
    for c, its in enumerate(items):
        for it in its:
            if it["kind"] != OWNER:
                continue
            owners += 1
            parts = partial_of.pop(it["tile"])
            assert [p[0] for p in parts] == list(range(c + 1, c + 1 + it["partners"]))
            edges = [it["kb1"]] + [p[2] for p in parts]
            assert [p[1] for p in parts] == edges[:-1] and edges[-1] == kb   # k order, no gap
    assert not partial_of                              # every partial piece has an owner
    if split_tiles == 0:
        assert owners == 0


def check_balance_and_coordinates(pl, items, tile_coord=g.tile_coord):
    """Stream-K ranges balanced to one k-block; coordinates are the raster's."""
    sk = [sum(it["kb1"] - it["kb0"] for it in its if it["tile"] < pl["sk_tiles"]) for its in items]
    if pl["sk_tiles"]:
        assert max(sk) - min(sk) <= 1
        assert sum(sk) == pl["sk_tiles"] * pl["k_blocks"]
    for its in items:
        for it in its:
            if pl["kernel"] == 1:      # the small-problem kernel: column-major tile order
                assert (it["m_tile"], it["n_tile"]) == (it["tile"] % pl["m_tiles"], it["tile"] // pl["m_tiles"])
                continue
            assert (it["m_tile"], it["n_tile"]) == tile_coord(it["tile"], pl["m_tiles"], pl["n_tiles"],
                                                              pl["swizzle"])


def check_small(pl, items):
    """The small-problem kernel: one item per cluster; with s = split_pieces
    pieces a tile, cluster c runs piece c % s of tile c // s over an equal share
    of the k-blocks, piece 0 owning the tile (adding the s - 1 clusters after it)
    and the others writing partials; without split-K every cluster is one whole
    tile."""
    if pl["kernel"] != 1:
        return
    s, kb = pl["split_pieces"], pl["k_blocks"]
    assert pl["clusters"] == pl["num_tiles"] * s and pl["grid_ctas"] == pl["clusters"] * pl["cta_group"]
    assert pl["tile_m"] == 128 * pl["cta_group"] and pl["tile_n"] in (32, 64, 128)
    assert (pl["sk_tiles"], pl["tail_split"]) == (0, 1) and (pl["workspace_bytes"] > 0) == (s > 1)
    assert s in (1, 2, 4, 8) and (s == 1 or kb // s >= 8)
    for c, its in enumerate(items):
        assert len(its) == 1
        it = its[0]
        t, pc = c // s, c % s
        kind = WHOLE if s == 1 else (OWNER if pc == 0 else PARTIAL)
        partners = s - 1 if s > 1 and pc == 0 else 0
        assert (it["tile"], it["kb0"], it["kb1"], it["kind"], it["parts"], it["partners"]) == \
            (t, kb * pc // s, kb * (pc + 1) // s, kind, 1, partners)


def check_k_order(pl, items):
    """The order in which the producer loads an item's k-blocks (k_down).  A
    partial piece loads from its last k-block down; an owner, a split piece and
    a stream-K piece covering a whole tile load up.  The whole tiles after the
    stream-K region go wave by wave (a cluster's j-th of them is in wave j):
    with plan k_order 0 all load up; with k_order 1 the first wave loads up
    and the direction flips every wave, the same for every cluster."""
    if pl["kernel"] == 1:
        assert all(it["k_down"] == 0 for its in items for it in its)
        return
    for its in items:
        j = 0
        for it in its:
            if it["kind"] == PARTIAL:
                assert it["k_down"] == 1, it
            elif it["kind"] in (OWNER, SPLIT) or it["tile"] < pl["sk_tiles"]:
                assert it["k_down"] == 0, it
            elif it["parts"] == 1:
                assert it["k_down"] == (j % 2 if pl["k_order"] else 0), (j, it)
                j += 1


def check_schedule(pl, items, tile_coord=g.tile_coord):
    check_small(pl, items)
    check_coverage(pl, items)
    check_partials_and_owners(pl, items)
    check_balance_and_coordinates(pl, items, tile_coord)
    check_k_order(pl, items)


@pytest.mark.parametrize("M,N,K,opts,mc", CASES, ids=lambda v: str(v))
def test_every_unit_exactly_once(M, N, K, opts, mc):
    check_coverage(*_all_items(M, N, K, opts, mc))


@pytest.mark.parametrize("M,N,K,opts,mc", CASES, ids=lambda v: str(v))
def test_partial_pieces_and_owners(M, N, K, opts, mc):
    check_partials_and_owners(*_all_items(M, N, K, opts, mc))


@pytest.mark.parametrize("M,N,K,opts,mc", CASES, ids=lambda v: str(v))
def test_stream_k_balance_and_coordinates(M, N, K, opts, mc):
    check_balance_and_coordinates(*_all_items(M, N, K, opts, mc))


@pytest.mark.parametrize("M,N,K,opts,mc", CASES, ids=lambda v: str(v))
def test_k_order_of_items(M, N, K, opts, mc):
    check_k_order(*_all_items(M, N, K, opts, mc))


@pytest.mark.parametrize("M,N,K,opts,mc,k_order", [
    (8192, 8192, 8192, {}, 76, 1),                   # a round's strips: 10 + 8 of 256 x 8192 = 75 MB
    (16384, 14336, 4096, {}, 76, 0),                 # 38 MB: forward only
    (4096, 4096, 4096, {}, 76, 0),
    (4000, 3000, 5000, {}, 76, 0),                   # 46 MB
    (4096, 4096, 16384, {}, 76, 1),
    (1024, 2048, 16384, {"cta_group": 2}, 16, 1),    # 2 + 8 strips of 256 x 16384 = 84 MB, two rounds
    (1024, 2048, 16384, {"cta_group": 2}, 32, 0),    # one round only: nothing to alternate
    (8192, 8192, 8192, {"accumulate": 1}, 76, 0),    # an fp16 accumulator keeps k order
])
def test_plan_k_order(M, N, K, opts, mc, k_order):
    assert g.plan(M, N, K, max_clusters=mc, options=g.Options(**opts))["k_order"] == k_order


@pytest.mark.parametrize("M,N,K,opts,mc,claimed", [
    (8192, 8192, 8192, {}, 76, 1024 % 76),           # 13 rounds dealt, the last 36 tiles claimed
    (16384, 14336, 4096, {}, 76, 3584 % 76),
    (4096, 4096, 4096, {}, 76, 0),                   # stream-K takes the last wave
    (4096, 4096, 4096, {"schedule": 1}, 76, 256 % 76),   # whole tiles only: 28 claimed
    (1100, 2100, 520, {"cta_group": 2, "schedule": 1}, 7, 45 % 7),
    (1024, 1024, 8192, {"cta_group": 2}, 64, 0),     # split pieces
    (2048, 2048, 1024, {"cta_group": 2, "schedule": 1}, 76, 0),  # 64 tiles: one wave, nothing left over
    (8192, 8192, 8192, {"schedule": 3}, 76, 0),      # N-split tail instead
    (700, 900, 1000, {"cta_group": 1, "schedule": 1}, 5, 24 % 5),
])
def test_plan_claimed_tiles(M, N, K, opts, mc, claimed):
    pl = g.plan(M, N, K, max_clusters=mc, options=g.Options(**opts))
    assert pl["claimed_tiles"] == claimed
    assert claimed < pl["clusters"]
    if claimed:
        assert (pl["sk_tiles"], pl["tail_split"], pl["split_pieces"]) == (0, 1, 1)
        assert pl["num_tiles"] > pl["clusters"]


def test_claimed_tiles_listed_in_cluster_order():
    """The schedule helper lists the claimed tiles as if cluster c took the c-th:
    each of the first claimed_tiles clusters ends on one tile of the last wave,
    the others end on their last dealt tile."""
    pl, items = _all_items(4096, 4096, 4096, {"schedule": 1}, 76)
    rem, G, T = pl["claimed_tiles"], pl["clusters"], pl["num_tiles"]
    assert rem == 256 % 76
    for c, its in enumerate(items):
        dealt = [it["tile"] for it in its if it["tile"] < T - rem]
        assert dealt == list(range(c, T - rem, G))
        last = [it["tile"] for it in its if it["tile"] >= T - rem]
        assert last == ([T - rem + c] if c < rem else [])


def test_n_split_tail_keeps_the_whole_tile_k_order():
    """A tile cut into column slices loads its k-blocks in the order it has as a
    whole tile, so that the two schedules give bit-identical results."""
    M = N = K = 8192
    split = _all_items(M, N, K, {"schedule": 3}, 76)
    whole = _all_items(M, N, K, {"schedule": 1}, 76)
    assert split[0]["tail_split"] > 1 and split[0]["k_order"] == whole[0]["k_order"] == 1
    down_whole = {it["tile"]: it["k_down"] for its in whole[1] for it in its}
    tail = [it for its in split[1] for it in its if it["parts"] > 1]
    assert tail and {it["k_down"] for it in tail} <= {0, 1}
    for it in tail:
        assert it["k_down"] == down_whole[it["tile"]], it


def test_schedule_rejects_a_cluster_out_of_range():
    pl = g.plan(4096, 4096, 4096, max_clusters=76)
    with pytest.raises(g.GemmError):
        g.schedule(4096, 4096, 4096, pl["clusters"], max_clusters=76)
    with pytest.raises(g.GemmError):
        g.schedule(4096, 4096, 4096, -1, max_clusters=76)
