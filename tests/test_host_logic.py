"""Host-side logic of the C-ABI library, on the CPU (no GPU needed).

Covers: every function declared in include/*.h is exported; the tile raster is a
bijection and reproduces the tutorial's worked wave example; the multiply-shift
division; the launch plan; argument validation returns its error codes before
any device work.
"""
import os
import re

import numpy as np
import pytest

import dense_fp16_gemm_gb300 as g

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    inc = os.path.join(ROOT, "include")
    for fn in os.listdir(inc):
        if fn.endswith(".h"):
            text = open(os.path.join(inc, fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(gemm_f16_nt\w*)\s*\(", text))
    return sorted(names)


def test_library_exports_every_declared_symbol():
    lib = g.library()
    names = declared_functions()
    assert "gemm_f16_nt" in names and len(names) >= 7, names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_status_strings():
    lib = g.library()
    for code, name in g.STATUS.items():
        assert lib.gemm_f16_nt_status_string(code).decode().startswith(name)
    assert b"unknown" in lib.gemm_f16_nt_status_string(99)


# ---------------------------------------------------------------------------
# scheduler
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("d", list(range(1, 300)) + [1000, 4095, 4096, 4097, 65535, 65536,
                                                      (1 << 30) - 1, 1 << 30, (1 << 30) + 1,
                                                      (1 << 31) - 1, 1 << 31])
def test_fast_divmod(d):
    rng = np.random.default_rng(d)
    ns = list(range(0, 2000)) + [(1 << 31) - 1, (1 << 31) - 2, d - 1, d, d + 1, 2 * d - 1, 2 * d]
    ns += [int(x) for x in rng.integers(0, 1 << 31, 300)]
    for n in ns:
        if n < 0 or n >= (1 << 31):
            continue
        assert g.fast_divmod(n, d) == divmod(n, d), (n, d)


def test_fast_divmod_rejects_out_of_range():
    with pytest.raises(g.GemmError):
        g.fast_divmod(5, 0)
    with pytest.raises(g.GemmError):
        g.fast_divmod(1 << 31, 3)


@pytest.mark.parametrize("sw", [1, 2, 3, 4, 5, 8, 16, 64])
def test_raster_is_bijection(sw):
    for mt in range(1, 21):
        for nt in range(1, 21):
            seen = set()
            for t in range(mt * nt):
                m, n = g.tile_coord(t, mt, nt, sw)
                assert 0 <= m < mt and 0 <= n < nt
                seen.add((m, n))
            assert len(seen) == mt * nt, (mt, nt, sw)


def test_raster_groups_are_row_major_with_narrow_last_group():
    # 5 x 7 grid, groups of 3 columns: groups {0,1,2}, {3,4,5}, {6} (narrower);
    # the odd group takes its rows from the bottom up
    order = [g.tile_coord(t, 5, 7, 3) for t in range(35)]
    assert order[:6] == [(0, 0), (0, 1), (0, 2), (1, 0), (1, 1), (1, 2)]
    assert order[15:21] == [(4, 3), (4, 4), (4, 5), (3, 3), (3, 4), (3, 5)]
    assert order[27:30] == [(0, 3), (0, 4), (0, 5)]
    assert order[30:] == [(0, 6), (1, 6), (2, 6), (3, 6), (4, 6)]


@pytest.mark.parametrize("mt,nt,sw", [(32, 32, 8), (64, 56, 8), (7, 20, 3), (9, 5, 2)])
def test_raster_groups_meet_on_the_same_rows(mt, nt, sw):
    # serpentine: the last tile of a group and the first of the next share a row
    order = [g.tile_coord(t, mt, nt, sw) for t in range(mt * nt)]
    starts = [t for t in range(1, mt * nt) if order[t][1] // sw != order[t - 1][1] // sw]
    assert starts
    for t in starts:
        assert order[t][0] == order[t - 1][0], (t, order[t - 1], order[t])


def test_raster_reproduces_the_pages_wave_example():
    path = os.path.join(ROOT, "tests", "golden", "raster_wave_8x8.txt")
    rows = [l.split() for l in open(path) if l.strip() and not l.startswith("#")]
    assert len(rows) == 2
    for r in rows:
        mt, nt, wave, sw, a_rows, b_cols, strips = map(int, r)
        tiles = [g.tile_coord(t, mt, nt, sw) for t in range(wave)]
        am = {m for m, _ in tiles}
        bn = {n for _, n in tiles}
        assert (len(am), len(bn), len(am) + len(bn)) == (a_rows, b_cols, strips)


def test_plan_headline_shape():
    p = g.plan(8192, 8192, 8192, num_sms=152)
    assert (p["cta_group"], p["tile_m"], p["tile_n"], p["block_k"]) == (2, 256, 256, 64)
    assert (p["m_tiles"], p["n_tiles"], p["k_blocks"], p["num_tiles"]) == (32, 32, 128, 1024)
    assert (p["clusters"], p["grid_ctas"]) == (76, 152)
    assert p["smem_bytes"] <= 232448 and p["tmem_cols"] == 512
    # 1024 tiles over 76 pairs: 13.47 rounds, the last one 47% full
    assert abs(p["num_tiles"] / p["clusters"] - 13.47) < 0.01


def test_plan_stream_k_schedule():
    # 4096^3: 256 tiles over 76 pairs leave 48 of 304 slots (16 %) idle: the
    # last wave (28 tiles) plus one full wave is split in k over all pairs
    p = g.plan(4096, 4096, 4096, num_sms=152)
    assert p["sk_tiles"] == 28 + 76 and p["tail_split"] == 1
    assert p["workspace_bytes"] == 76 * 2 * 4 * 8 + 76 * 2 * 128 * 256 * 4
    # ... only for deep k (each cluster spared >= 32 k-blocks) and with a full
    # wave of whole tiles left; shallow last waves take the N-split instead
    assert g.plan(6144, 4096, 4096, num_sms=152)["sk_tiles"] == 4 + 76
    assert g.plan(4096, 11008, 4096, num_sms=152)["sk_tiles"] == 4 + 76   # 9.5 % of slots idle
    pers = g.Options(cta_group=2)                         # the persistent kernel (small problems
    # default to the small-problem kernel; test_plan_small_kernel)
    p = g.plan(512, 4096, 4096, num_sms=152, options=pers)  # 32 tiles of 64 k-blocks: two split pieces each
    assert (p["sk_tiles"], p["tail_split"], p["split_pieces"], p["clusters"]) == (0, 1, 2, 64)
    p = g.plan(4096, 4096, 1024, num_sms=152)             # 16 k-blocks
    assert (p["sk_tiles"], p["tail_split"], p["tail_tiles"]) == (0, 2, 28)
    p = g.plan(3584, 2304, 2048, num_sms=152)             # 32 k-blocks, 126 tiles
    assert (p["sk_tiles"], p["tail_split"]) == (0, 1)
    p = g.plan(2048, 4096, 8192, num_sms=152)             # 128 tiles: no full wave would stay whole
    assert (p["sk_tiles"], p["tail_split"]) == (0, 1)
    # 8192^3: 40 of 1064 slots (3.8 %) idle: whole tiles, unless forced
    assert g.plan(8192, 8192, 8192, num_sms=152)["sk_tiles"] == 0
    assert g.plan(8192, 8192, 8192, num_sms=152)["tail_split"] == 1
    assert g.plan(8192, 8192, 8192, options=g.Options(schedule=2))["sk_tiles"] == 36 + 76
    # whole tiles only on request, or when the last wave is nearly full
    p = g.plan(4096, 4096, 4096, options=g.Options(schedule=1))
    assert (p["sk_tiles"], p["workspace_bytes"], p["tail_split"]) == (0, 0, 1)
    p = g.plan(256 * 19, 256 * 8, 4096, num_sms=152)      # 152 tiles = 2 full waves
    assert (p["sk_tiles"], p["tail_split"]) == (0, 1)
    p = g.plan(256 * 15, 256 * 10, 4096, num_sms=152)     # 150 tiles: last wave 74/76 full
    assert (p["sk_tiles"], p["tail_split"]) == (0, 1)
    # fewer tiles than pairs and deep k (>= 48 k-blocks): every tile cut into
    # s = 2, 4 or 8 split pieces, the largest with tiles * s <= pairs
    one = g.Options(cluster_pairs=1, cta_group=2)
    p = g.plan(1024, 1024, 8192, options=one)             # 16 tiles x 128 k-blocks: 4 pieces
    assert (p["sk_tiles"], p["split_pieces"], p["clusters"], p["tail_split"]) == (0, 4, 64, 1)
    assert p["workspace_bytes"] == 64 * 2 * 4 * 8 + 64 * 2 * 128 * 256 * 4
    p = g.plan(256, 256, 8192, options=one)               # 1 tile x 128 k-blocks: 8 pieces
    assert (p["split_pieces"], p["clusters"]) == (8, 8)
    p = g.plan(1024, 1024, 1024, options=one)             # 16 x 16 k-blocks: too shallow, N-split
    assert (p["split_pieces"], p["tail_split"], p["clusters"]) == (1, 4, 64)
    p = g.plan(2048, 2048, 2048, options=one)             # 64 tiles: no room for 2 pieces each
    assert (p["split_pieces"], p["clusters"]) == (1, 64)
    p = g.plan(1000, 700, 1000, options=one)              # 12 x 16 k-blocks: N-split
    assert (p["split_pieces"], p["clusters"], p["tail_split"]) == (1, 48, 4)
    # forced (schedule 4): from one k-block a piece; never for an fp16 accumulator
    p = g.plan(300, 520, 328, options=g.Options(schedule=4))
    assert (p["split_pieces"], p["clusters"]) == (4, 24)
    assert g.plan(256, 256, 8192, options=g.Options(schedule=4, accumulate=1))["split_pieces"] == 1
    assert g.plan(256, 256, 8192, options=g.Options(schedule=1))["split_pieces"] == 1
    # the owner-based stream-K split over all tiles stays available when forced
    p = g.plan(256, 256, 4096, options=g.Options(schedule=2))   # forced: one k-block per pair
    assert (p["sk_tiles"], p["clusters"], p["split_pieces"]) == (1, 64, 1)
    with pytest.raises(g.GemmError):
        g.plan(256, 256, 256, options=g.Options(schedule=6))


def test_plan_n_split():
    # fewer tiles than pairs and too few k-blocks for stream-K: each tile is cut
    # along N into s = 2 or 4 slices, the largest with tiles·s <= pairs
    pers = g.Options(cta_group=2)                         # the persistent kernel
    p = g.plan(256, 256, 256, options=pers)               # 1 tile x 4 k-blocks
    assert (p["tail_tiles"], p["tail_split"], p["clusters"], p["grid_ctas"], p["sk_tiles"]) == (1, 4, 4, 8, 0)
    p = g.plan(300, 520, 328, options=g.Options(cluster_pairs=1, cta_group=2))   # 6 tiles x 6 k-blocks
    assert (p["tail_tiles"], p["tail_split"], p["clusters"]) == (6, 4, 24)
    p = g.plan(256 * 6, 256 * 5, 256, options=pers)       # 30 tiles: 30·2 <= 76 < 30·4
    assert (p["tail_tiles"], p["tail_split"], p["clusters"]) == (30, 2, 60)
    # not for full waves (a narrower MMA is not faster per k-block), unless forced (3)
    for shape in ((8192, 8192, 8192), (16384, 14336, 4096)):
        assert g.plan(*shape, num_sms=152)["tail_split"] == 1
    p = g.plan(8192, 8192, 8192, options=g.Options(schedule=3))
    assert (p["tail_tiles"], p["tail_split"], p["sk_tiles"], p["clusters"]) == (36, 2, 0, 76)
    p = g.plan(16384, 14336, 4096, options=g.Options(schedule=3))
    assert (p["tail_tiles"], p["tail_split"]) == (12, 4)
    assert g.plan(256 * 15, 256 * 10, 4096, options=g.Options(schedule=3))["tail_split"] == 1   # R = 74
    # not with two pairs per cluster, one CTA, B stored [K, N], or another forced schedule
    mc = g.library_mcast()
    assert g.plan(256, 256, 256, options=g.Options(cluster_pairs=2), lib=mc)["tail_split"] == 1
    for o in (g.Options(cta_group=1), g.Options(b_layout=1), g.Options(schedule=1), g.Options(schedule=2)):
        assert g.plan(256, 256, 256, options=o)["tail_split"] == 1
    # the fp16 accumulator may use it (each output's sum is unchanged)
    assert g.plan(256, 256, 256, options=g.Options(accumulate=1))["tail_split"] == 4


def test_plan_two_pairs_per_cluster():
    # only the single-GPU multicast build has two pairs per cluster
    o = g.Options(cluster_pairs=2)
    with pytest.raises(g.GemmError):
        g.plan(8192, 8192, 8192, num_sms=152, max_clusters=36, options=o)
    mc = g.library_mcast()
    assert (mc.gemm_f16_nt_multicast_available(), g.library().gemm_f16_nt_multicast_available()) == (1, 0)
    p = g.plan(8192, 8192, 8192, num_sms=152, max_clusters=36, options=o, lib=mc)
    assert (p["cluster_pairs"], p["tile_m"], p["tile_n"]) == (2, 256, 512)
    assert (p["m_tiles"], p["n_tiles"], p["num_tiles"]) == (32, 16, 512)
    assert (p["clusters"], p["grid_ctas"]) == (36, 144)
    assert p["sk_tiles"] == 0                           # auto: two pairs keep whole tiles
    o = g.Options(cluster_pairs=2, schedule=2)
    p = g.plan(8192, 8192, 8192, num_sms=152, max_clusters=36, options=o, lib=mc)
    assert p["sk_tiles"] == 512 % 36 + 36               # forced: last wave 8/36 + one wave
    assert p["workspace_bytes"] == 36 * 4 * 4 * 8 + 36 * 4 * 128 * 256 * 4
    p = g.plan(4000, 3000, 5000, num_sms=152, max_clusters=36, options=o, lib=mc)
    assert (p["m_tiles"], p["n_tiles"]) == (16, 6)
    # K = 5000: 10,000-byte rows are not 128-byte multiples, so the multicast
    # build's default shares A between two pairs (256 x 512 cluster tiles);
    # the default build keeps one pair
    p = g.plan(4000, 3000, 5000, lib=mc)
    assert (p["cluster_pairs"], p["m_tiles"], p["n_tiles"]) == (2, 16, 6)
    assert g.plan(8192, 8192, 8192, lib=mc)["cluster_pairs"] == 1
    assert g.plan(4000, 256, 5000, lib=mc)["cluster_pairs"] == 1      # too narrow for two pairs
    for lib in (mc, g.library()):
        with pytest.raises(g.GemmError):
            g.plan(256, 256, 256, options=g.Options(cluster_pairs=2, cta_group=1), lib=lib)
        with pytest.raises(g.GemmError):
            g.plan(256, 256, 256, options=g.Options(cluster_pairs=3), lib=lib)


def test_plan_edges_and_options():
    p = g.plan(4000, 3000, 5000, options=g.Options(cluster_pairs=1))
    assert (p["m_tiles"], p["n_tiles"], p["k_blocks"]) == (16, 12, 79)
    # the default build has one pair per cluster for every pitch
    p = g.plan(4000, 3000, 5000)
    assert (p["cluster_pairs"], p["m_tiles"], p["n_tiles"]) == (1, 16, 12)
    p = g.plan(100, 100, 8, options=g.Options(cta_group=2))   # one pair tile, rank-1 rows all out of range,
    # cut into four 64-column slices (the last two lie wholly past N and store nothing)
    assert (p["num_tiles"], p["clusters"], p["grid_ctas"], p["tail_split"]) == (1, 4, 8, 4)
    p = g.plan(100, 100, 8, options=g.Options(schedule=1))
    assert (p["num_tiles"], p["clusters"], p["grid_ctas"]) == (1, 1, 2)
    p1 = g.plan(4000, 3000, 5000, options=g.Options(cta_group=1))
    assert (p1["tile_m"], p1["m_tiles"], p1["grid_ctas"]) == (128, 32, 152)
    p = g.plan(8192, 8192, 8192, options=g.Options(max_clusters=3, swizzle=4))
    assert (p["clusters"], p["swizzle"]) == (3, 4)
    p = g.plan(8192, 300, 64, options=g.Options(swizzle=16))
    assert p["swizzle"] == 2                         # clipped to the 2 N tiles
    for bad in (g.Options(cta_group=3), g.Options(swizzle=65), g.Options(max_clusters=-1)):
        with pytest.raises(g.GemmError):
            g.plan(256, 256, 256, options=bad)
    with pytest.raises(g.GemmError):
        g.plan(-1, 5, 5)
    with pytest.raises(g.GemmError):
        g.plan(1 << 31, 5, 5)


# ---------------------------------------------------------------------------
# argument validation (returns before any CUDA call)
# ---------------------------------------------------------------------------

def call(M, N, K, a=0x10000, lda=None, b=0x20000, ldb=None, c=0x30000, ldc=None, opts=None):
    lib = g.library()
    lda = K if lda is None else lda
    ldb = K if ldb is None else ldb
    ldc = N if ldc is None else ldc
    if opts is None:
        return lib.gemm_f16_nt(M, N, K, a, lda, b, ldb, c, ldc, None)
    return lib.gemm_f16_nt_ex(M, N, K, a, lda, b, ldb, c, ldc, None, opts)


@pytest.mark.parametrize("args,code", [
    (dict(M=-1, N=8, K=8), 1),
    (dict(M=8, N=8, K=1 << 31), 1),
    (dict(M=8, N=8, K=16, lda=8), 1),               # lda < K
    (dict(M=8, N=8, K=16, ldb=8), 1),               # ldb < K
    (dict(M=8, N=16, K=16, ldc=8), 1),              # ldc < N
    (dict(M=8, N=8, K=16, a=0), 1),                 # NULL A
    (dict(M=8, N=8, K=16, c=0), 1),                 # NULL C
    (dict(M=8, N=8, K=16, a=0x10008), 2),           # A not 16-byte aligned
    (dict(M=8, N=8, K=16, b=0x20002), 2),
    (dict(M=8, N=8, K=16, c=0x30004), 2),
    (dict(M=8, N=8, K=12, lda=12, ldb=16), 2),      # lda not a multiple of 8
    (dict(M=8, N=12, K=16, ldc=12), 2),             # ldc not a multiple of 8
    (dict(M=0, N=8, K=16, a=0, b=0, c=0), 0),       # empty output: no-op
    (dict(M=8, N=0, K=16), 0),
])
def test_argument_validation(args, code):
    assert call(**args) == code


def test_layout_pitches_validated():
    # A stored [K, M]: lda counts M; B stored [K, N]: ldb counts N
    assert call(64, 32, 16, lda=32, ldb=16, opts=g.Options(a_layout=1)) == 1     # lda < M
    assert call(16, 64, 40, lda=40, ldb=32, opts=g.Options(b_layout=1)) == 1     # ldb < N
    assert call(16, 64, 36, lda=36, ldb=64, ldc=64, opts=g.Options(b_layout=1)) == 2     # lda % 8 != 0
    assert call(8, 8, 16, opts=g.Options(a_layout=2)) == 1
    assert call(8, 8, 16, opts=g.Options(accumulate=2)) == 1


def test_fp16_accumulation_option_validated():
    lib = g.library()
    # fp16 accumulator with bf16 operands: rejected before anything is enqueued
    assert lib.gemm_bf16_nt_ex(8, 8, 16, 0x10000, 16, 0x20000, 16, 0x30000, 8, None,
                               g.Options(accumulate=1)) == 1
    assert call(8, 8, 16, opts=g.Options(accumulate=-1)) == 1
    # the fp16 accumulator never splits in k
    assert g.plan(4096, 4096, 4096, options=g.Options(accumulate=1))["sk_tiles"] == 0
    assert g.plan(4096, 4096, 4096, options=g.Options(accumulate=1, schedule=2))["sk_tiles"] == 0
    assert g.plan(256, 256, 8192, options=g.Options(accumulate=1, schedule=1))["clusters"] == 1


def test_bad_options_rejected():
    assert call(8, 8, 16, opts=g.Options(cta_group=4)) == 1
    assert call(8, 8, 16, opts=g.Options(swizzle=-1)) == 1
    assert call(8, 8, 16, opts=g.Options(schedule=7)) == 1


def test_without_a_gpu_valid_calls_report_no_device():
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present; this case is for GPU-less hosts")
    assert call(128, 128, 64) == 3
    assert g.library().gemm_f16_nt_device_status(None, None) == 3


def test_noalloc_scratch_limit_condition():
    """gemm_f16_nt_noalloc keeps its stream-K scratch in a fixed 20 MiB array and
    rejects (GEMM_ERR_SCRATCH_LIMIT) a plan whose workspace exceeds it.  On a
    152-SM GB300 no plan does; on a GPU with more SMs the same shape would."""
    limit = 20 << 20
    for sms in (148, 152):
        for shape in ((4096, 4096, 4096), (6144, 4096, 4096), (1024, 1024, 8192), (256, 256, 1 << 20)):
            for o in (g.Options(), g.Options(schedule=2), g.Options(cta_group=1, schedule=2)):
                assert g.plan(*shape, num_sms=sms, options=o)["workspace_bytes"] <= limit
    big = g.plan(4096, 4096, 4096, num_sms=176, options=g.Options(schedule=2))
    assert big["workspace_bytes"] > limit


def test_plan_small_kernel():
    # problems whose 128-row tiles fit on the SMs in one wave take the small-
    # problem kernel: one CTA per 128 x bn tile, bn the narrowest of 32, 64, 128
    # that fits, all of k in one CTA
    for (M, N, K), (bn, tiles) in {(256, 256, 256): (32, 16), (64, 64, 64): (32, 2), (1024, 1024, 1024): (64, 128),
                                   (512, 4096, 4096): (128, 128), (128, 4096, 4096): (32, 128),
                                   (768, 768, 2048): (32, 144), (1000, 1000, 1000): (64, 128),
                                   (1024, 1024, 8192): (64, 128)}.items():
        p = g.plan(M, N, K, num_sms=152)
        assert (p["kernel"], p["cta_group"], p["tile_m"], p["tile_n"]) == (1, 1, 128, bn), (M, N, K)
        assert (p["num_tiles"], p["clusters"], p["grid_ctas"]) == (tiles, tiles, tiles), (M, N, K)
        assert (p["sk_tiles"], p["split_pieces"], p["tail_split"], p["workspace_bytes"]) == (0, 1, 1, 0)
        assert p["k_blocks"] == -(-K // 64) and p["smem_bytes"] <= 232448
        assert p["tmem_cols"] == max(32, bn)
    # few tiles and deep k: split-K, s pieces a tile (s <= 8, a power of two, all
    # pieces in one wave, >= 8 k-blocks a piece); piece 0 owns the tile
    for (M, N, K), (bn, tiles, s) in {(256, 256, 4096): (32, 16, 8), (256, 256, 1 << 16): (32, 16, 8),
                                      (512, 512, 8192): (32, 64, 2), (300, 200, 3000): (32, 21, 4),
                                      (256, 256, 1024): (32, 16, 1), (256, 256, 2048): (32, 16, 4), (100, 100, 600): (32, 4, 1)}.items():
        p = g.plan(M, N, K, num_sms=152)
        assert (p["kernel"], p["tile_n"], p["num_tiles"], p["split_pieces"]) == (1, bn, tiles, s), (M, N, K)
        assert (p["clusters"], p["grid_ctas"], p["sk_tiles"], p["tail_split"]) == (tiles * s, tiles * s, 0, 1)
        # the workspace: per-warp flags (256-byte aligned), then one fp32 128 x bn partial per CTA
        flags = -(-tiles * s * 4 * 8 // 256) * 256
        assert p["workspace_bytes"] == (flags + tiles * s * 128 * bn * 4 if s > 1 else 0)
    # more than one wave, or more than 128 k-blocks a piece: the persistent kernel
    for M, N, K in ((2048, 2048, 2048), (4096, 1024, 1024), (8192, 8192, 8192), (256, 256, 1 << 17),
                    (1024, 1024, 8256)):
        assert g.plan(M, N, K, num_sms=152)["kernel"] == 0, (M, N, K)
    # the wave is counted on the given SM count
    assert g.plan(1024, 1024, 1024, num_sms=100)["tile_n"] == 128
    # any persistent-kernel option keeps the persistent kernel
    for o in (g.Options(cta_group=2), g.Options(cta_group=1), g.Options(swizzle=4), g.Options(max_clusters=8),
              g.Options(schedule=1), g.Options(schedule=3), g.Options(a_layout=1), g.Options(b_layout=1),
              g.Options(accumulate=1)):
        assert g.plan(256, 256, 256, options=o)["kernel"] == 0
    # forced (schedule 5): any shape, CTA group and tile width asked for
    p = g.plan(8192, 8192, 8192, options=g.Options(schedule=5))
    assert (p["kernel"], p["cta_group"], p["tile_n"], p["num_tiles"]) == (1, 1, 128, 64 * 64)
    p = g.plan(300, 520, 328, options=g.Options(schedule=5, cta_group=2, tile_n=64))
    assert (p["kernel"], p["cta_group"], p["tile_m"], p["tile_n"], p["m_tiles"], p["n_tiles"]) == (1, 2, 256, 64, 2, 9)
    assert (p["clusters"], p["grid_ctas"]) == (18, 36)
    for bad in (g.Options(schedule=5, tile_n=48), g.Options(schedule=5, tile_n=256), g.Options(tile_n=16),
                g.Options(schedule=5, a_layout=1), g.Options(schedule=5, b_layout=1),
                g.Options(schedule=5, accumulate=1)):
        with pytest.raises(g.GemmError):
            g.plan(256, 256, 256, options=bad)
    mc = g.library_mcast()
    with pytest.raises(g.GemmError):
        g.plan(256, 256, 256, options=g.Options(schedule=5, cluster_pairs=2), lib=mc)
    # the multicast build plans the same small-problem kernel
    assert g.plan(256, 256, 256, lib=mc)["kernel"] == 1
    # its schedule: cluster c computes tile c (column-major), all of k
    items = [g.schedule(300, 520, 328, c, options=g.Options(schedule=5, cta_group=2, tile_n=64)) for c in range(18)]
    assert [(it[0]["m_tile"], it[0]["n_tile"], it[0]["kb0"], it[0]["kb1"]) for it in items] == \
        [(c % 2, c // 2, 0, 6) for c in range(18)]
