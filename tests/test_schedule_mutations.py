"""The schedule checks must catch plausible mistakes in the schedule code.

The kernel's work schedule (sched.cuh: the raster, work_init / work_next,
owner_partners, set_schedule) is plain integer C++ that compiles for the host
too.  This file builds a small host library from a copy of sched.cuh (on the
CPU, in a temporary directory), enumerates every cluster's items for a set of
planned problems, and runs the checks of test_schedule.py on them:
  - the unchanged copy passes every check and gives exactly the items that
    gemm_f16_nt_schedule reports;
  - each copy with one planted mistake fails at least one check.
The committed sched.cuh is never modified.
"""
import ctypes
import os
import shutil
import subprocess
import tempfile

import pytest

import dense_fp16_gemm_gb300 as g
from dense_fp16_gemm_gb300 import _build_ext
import tests.test_schedule as ts

_SCHED = os.path.join(_build_ext.CSRC, "sched.cuh")

_HARNESS = r"""
#include <stdint.h>
#include "sched.cuh"

namespace {
struct Sp { uint32_t num_tiles, num_kb, sk_tiles; uint64_t sk_units; uint32_t tail_first, tail_split, split_pieces, k_alternate, dyn_first; };
struct Pl { int64_t num_tiles; int32_t k_blocks, sk_tiles, tail_split, tail_tiles, split_pieces, k_order, claimed_tiles; };
}

extern "C" int32_t sched_items(int64_t num_tiles, int32_t k_blocks, int32_t sk_tiles, int32_t tail_split,
                               int32_t tail_tiles, int32_t split_pieces, int32_t k_order, int32_t claimed_tiles,
                               int32_t m_tiles, int32_t n_tiles, int32_t swizzle, int32_t clusters, int32_t cluster,
                               int32_t* out, int32_t max_items) {
    Pl pl{num_tiles, k_blocks, sk_tiles, tail_split, tail_tiles, split_pieces, k_order, claimed_tiles};
    Sp sp;
    g16::set_schedule(sp, pl);
    const g16::Raster r = g16::make_raster(uint32_t(m_tiles), uint32_t(n_tiles), uint32_t(swizzle));
    g16::Work w;
    g16::Item it;
    g16::work_init(w, sp, uint32_t(cluster), uint32_t(clusters));
    int32_t n = 0;
    while (g16::work_next(w, sp, it)) {
        if (n < max_items) {
            uint32_t mt, nt;
            g16::raster_coord(r, it.tile, mt, nt);
            int32_t* o = out + 12 * n;
            o[0] = int32_t(it.tile); o[1] = int32_t(mt); o[2] = int32_t(nt);
            o[3] = int32_t(it.kb0); o[4] = int32_t(it.kb1); o[5] = int32_t(it.kind);
            o[6] = int32_t(it.part); o[7] = int32_t(it.parts);
            o[8] = it.kind == g16::kItemOwner
                       ? int32_t(g16::owner_partners(sp, it.tile, uint32_t(cluster), uint32_t(clusters))) : 0;
            o[9] = int32_t(it.piece); o[10] = int32_t(it.pieces);
            o[11] = int32_t(g16::item_k_down(sp, it, uint32_t(clusters)));
        }
        if (++n >= (1 << 20)) return -1;   // a schedule that never ends
    }
    return n;
}
"""

_FIELDS = ("tile", "m_tile", "n_tile", "kb0", "kb1", "kind", "part", "parts", "partners", "piece", "pieces",
           "k_down")

# M, N, K, options, max_clusters: stream-K (last wave, forced, few tiles with
# middle pieces), N-split (small problem, forced tail), two pairs, cta_group 1
CASES = [
    (4096, 4096, 4096, {}, 76),
    (8192, 8192, 8192, {"schedule": 2}, 76),
    (8192, 8192, 8192, {"schedule": 3}, 76),
    (256, 256, 256, {"cta_group": 2}, 76),            # (the persistent kernel: small problems
    (256, 256, 8192, {"cta_group": 2}, 76),           #  default to the small-problem kernel)
    (1024, 1024, 8192, {"cta_group": 2}, 64),
    (4096, 4096, 1024, {}, 76),
    (4000, 3000, 5000, {}, 36),
    (1300, 1000, 320, {"schedule": 3, "cluster_pairs": 1}, 76),
    (700, 900, 1000, {"cta_group": 1, "schedule": 2}, 152),
    (6000, 7000, 3000, {}, 76),
    (300, 520, 328, {"schedule": 4}, 76),             # split pieces of 1 or 2 k-blocks
    (256, 256, 8192, {"schedule": 4}, 76),            # one tile in 8 pieces
    (8192, 8192, 8192, {}, 76),                       # whole tiles, k order alternating by round
    (1024, 2048, 16384, {"cta_group": 2}, 16),        # two rounds, k order alternating
    (1024, 2048, 16384, {"cta_group": 2, "schedule": 2}, 12),   # stream-K, then alternating rounds
]
assert all(g.plan(M, N, K, max_clusters=mc, options=g.Options(**o))["kernel"] == 0 for M, N, K, o, mc in CASES)

MUTATIONS = {
    "stream_k_ranges_rounded_per_cluster": ("return p.sk_units * c / G;", "return p.sk_units / G * c;"),
    "whole_tiles_start_at_zero": ("s.t = p.sk_tiles + c;", "s.t = c;"),
    "owner_counts_a_partner_starting_at_the_tile_end": (
        "sk_begin(p, c + 1 + n, G) < tile_end", "sk_begin(p, c + 1 + n, G) <= tile_end"),
    "owner_counts_itself": (
        "while (c + 1 + n < G && sk_begin(p, c + 1 + n, G) < tile_end) ++n;",
        "while (c + n < G && sk_begin(p, c + n, G) < tile_end) ++n;"),
    "every_slice_is_part_zero": ("it.part = s.q % p.tail_split;", "it.part = 0;"),
    "split_tail_dropped": (
        "p.tail_first = uint32_t(pl.num_tiles - (pl.tail_split > 1 ? pl.tail_tiles : 0));",
        "p.tail_first = uint32_t(pl.num_tiles);"),
    "serpentine_on_even_groups": ("m_tile = (g & 1u) ? r.m_tiles - 1u - mm : mm;",
                                  "m_tile = (g & 1u) ? mm : r.m_tiles - 1u - mm;"),
    "narrow_last_group_ignored": ("const FastDiv& w = (first_n + r.swizzle <= r.n_tiles) ? r.full : r.last;",
                                  "const FastDiv& w = r.full;"),
    "split_piece_ranges_rounded": ("it.kb0 = uint32_t(uint64_t(p.num_kb) * piece / np);",
                                   "it.kb0 = p.num_kb / np * piece;"),
    "split_piece_tile_from_remainder": ("it.tile = s.t / np;", "it.tile = s.t % np;"),
    "split_piece_index_from_quotient": ("const uint32_t np = p.split_pieces, piece = s.t % np;",
                                        "const uint32_t np = p.split_pieces, piece = s.t / np;"),
    "k_order_ignored": ("if (!p.k_alternate || it.kind != kItemWhole", "if (it.kind != kItemWhole"),
    "k_order_by_tile_parity": ("return (((it.tile - p.sk_tiles) / G) & 1u) != 0;", "return (it.tile & 1u) != 0;"),
    "k_order_in_even_rounds": ("return (((it.tile - p.sk_tiles) / G) & 1u) != 0;",
                               "return (((it.tile - p.sk_tiles) / G) & 1u) == 0;"),
    "stream_k_tiles_alternate": ("it.kind != kItemWhole || it.tile < p.sk_tiles", "it.kind != kItemWhole"),
    "claimed_tiles_also_dealt": ("if (s.t < p.tail_first && s.t < p.dyn_first) {", "if (s.t < p.tail_first) {"),
    "claim_asked_twice": ("        if (s.claimed) return false;\n", ""),
    "claimed_range_off_by_one": ("const uint32_t t = p.dyn_first + s.c;", "const uint32_t t = p.dyn_first + s.c + 1;"),
    "piece_kinds_swapped": (
        "it.kind = kb0 > 0 ? kItemPartialOut : (kb1 < p.num_kb ? kItemOwner : kItemWhole);",
        "it.kind = kb1 < p.num_kb ? kItemPartialOut : (kb0 > 0 ? kItemOwner : kItemWhole);"),
}


def _compiler():
    for c in ("g++", "c++"):
        if shutil.which(c):
            return c
    pytest.skip("no C++ compiler")


def _build(tmp, source):
    d = tempfile.mkdtemp(dir=tmp)
    with open(os.path.join(d, "sched.cuh"), "w") as f:
        f.write(source)
    with open(os.path.join(d, "harness.cpp"), "w") as f:
        f.write(_HARNESS)
    out = os.path.join(d, "libsched.so")
    subprocess.run([_compiler(), "-std=c++17", "-O1", "-shared", "-fPIC", "-I" + d, "-o", out,
                    os.path.join(d, "harness.cpp")], check=True, capture_output=True)
    lib = ctypes.CDLL(out)
    lib.sched_items.restype = ctypes.c_int32
    lib.sched_items.argtypes = [ctypes.c_int64] + [ctypes.c_int32] * 12 + [ctypes.POINTER(ctypes.c_int32),
                                                                            ctypes.c_int32]
    return lib


def _items(lib, pl):
    args = (pl["num_tiles"], pl["k_blocks"], pl["sk_tiles"], pl["tail_split"], pl["tail_tiles"],
            pl["split_pieces"], pl["k_order"], pl["claimed_tiles"], pl["m_tiles"], pl["n_tiles"], pl["swizzle"],
            pl["clusters"])
    out = []
    for c in range(pl["clusters"]):
        n = lib.sched_items(*args, c, None, 0)
        buf = (ctypes.c_int32 * (12 * max(n, 1)))()
        lib.sched_items(*args, c, buf, n)
        out.append([dict(zip(_FIELDS, buf[12 * i:12 * i + 12])) for i in range(n)])
    return out


def _plans():
    return [g.plan(M, N, K, max_clusters=mc, options=g.Options(**o)) for M, N, K, o, mc in CASES]


def _failures(lib):
    bad = []
    for case, pl in zip(CASES, _plans()):
        try:
            ts.check_schedule(pl, _items(lib, pl))
        except AssertionError:
            bad.append(case)
    return bad


def test_unchanged_copy_passes_and_matches_the_library(tmp_path):
    lib = _build(str(tmp_path), open(_SCHED).read())
    assert _failures(lib) == []
    for (M, N, K, o, mc), pl in zip(CASES, _plans()):
        mine = _items(lib, pl)
        theirs = [g.schedule(M, N, K, c, max_clusters=mc, options=g.Options(**o)) for c in range(pl["clusters"])]
        assert mine == theirs, (M, N, K, o)


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(tmp_path, name):
    old, new = MUTATIONS[name]
    src = open(_SCHED).read()
    assert src.count(old) == 1, f"mutation {name} no longer applies"
    lib = _build(str(tmp_path), src.replace(old, new))
    assert _failures(lib), f"no check caught the mutation {name}"
