"""The two builds of the library, checked on the CPU.

libgemm_f16_nt.so is the library every process loads, on any number of GPUs:
no source it is compiled from may issue a multicast copy (a cp.async.bulk
form with .multicast::cluster).  libgemm_f16_nt_mcast.so adds clusters of two
CTA pairs sharing A by TMA multicast; it is built from a separate translation
unit and is for single-GPU processes only.  Both export the whole C ABI.
"""
import os
import re

import pytest

import dense_fp16_gemm_gb300 as g
from dense_fp16_gemm_gb300 import _build_ext
from tests.test_host_logic import declared_functions

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def asm_statements(text: str):
    """The PTX text of every asm statement in a C++ source (its adjacent string
    literals joined), so that an instruction split over several literals is
    seen whole."""
    out = []
    for m in re.finditer(r"\basm\s+(?:volatile\s*)?\(", text):
        i, depth = m.end(), 1
        while depth and i < len(text):
            depth += {"(": 1, ")": -1}.get(text[i], 0)
            i += 1
        body = text[m.end():i - 1]
        # the template is the string literals before the first ':' outside a literal
        parts, j = [], 0
        while j < len(body) and body[j] != ":":
            if body[j] == '"':
                k = j + 1
                while body[k] != '"':
                    k += 2 if body[k] == "\\" else 1
                parts.append(body[j + 1:k])
                j = k
            j += 1
        out.append("".join(parts))
    return out


def test_default_build_sources_issue_no_multicast_copy():
    srcs = set(_build_ext.DEPENDS)
    for fn in os.listdir(_build_ext.CSRC):          # everything the default build can include
        if fn.endswith((".cu", ".cuh", ".h")):
            srcs.add(os.path.join(_build_ext.CSRC, fn))
    assert not any(os.sep + "mcast" + os.sep in p for p in srcs)
    seen_copies = 0
    for path in sorted(srcs):
        text = open(path).read()
        assert "tma_multicast.cuh" not in text, path
        for ptx in asm_statements(text):
            if "cp.async.bulk" in ptx:
                seen_copies += 1
                assert "multicast" not in ptx, f"{path}: multicast copy {ptx!r}"
    assert seen_copies >= 4        # the loads and the store are there, without multicast
    # the one default-source mention of `.multicast::cluster` is tcgen05.commit's
    # completion signal to the two CTAs of a pair (an mbarrier arrive, no data)
    for path in sorted(srcs):
        for ptx in asm_statements(open(path).read()):
            if "multicast" in ptx:
                assert ptx.startswith("tcgen05.commit"), (path, ptx)


def test_multicast_load_lives_only_in_the_opt_in_build():
    mc = [p for p in _build_ext.MCAST_DEPENDS if os.sep + "mcast" + os.sep in p]
    loads = [ptx for p in mc for ptx in asm_statements(open(p).read())
             if "cp.async.bulk" in ptx and "multicast" in ptx]
    assert len(loads) == 1
    # bench.py never names it either
    bench = open(os.path.join(ROOT, "bench.py")).read()
    assert ".multicast::cluster" not in bench


@pytest.mark.parametrize("variant", ["default", "mcast"])
def test_both_builds_export_the_c_abi(variant):
    lib = g.library(variant=variant)
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported by {variant}"
    assert lib.gemm_f16_nt_multicast_available() == (1 if variant == "mcast" else 0)


def test_default_build_refuses_two_pairs_per_cluster():
    from tests.test_host_logic import call
    assert call(512, 1024, 64, opts=g.Options(cluster_pairs=2)) == 1
    with pytest.raises(g.GemmError):
        g.plan(512, 1024, 64, options=g.Options(cluster_pairs=2))


def test_multicast_library_refused_in_a_multi_rank_process(monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "2")
    with pytest.raises(RuntimeError):
        g.library_mcast()
