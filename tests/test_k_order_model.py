"""The plan's k-order rule against the L2 model it rests on (tests/l2_model.py).

The plan alternates the k direction of odd whole-tile waves (k_order 1) when
a wave's A and B strips exceed 60 MB.  The model, fitted to measured DRAM
reads at 8192³, must agree: where the plan alternates, alternating reads
clearly fewer bytes; where it does not, alternating saves nothing worth it.
"""
import pytest

import dense_fp16_gemm_gb300 as g
from tests import l2_model


def test_model_reproduces_the_measured_raster_widths():
    """The fit the rule rests on: DRAM reads of the up-only order at 8192³ for
    group widths 4, 8 and 16 (measured on a GB300: 1.34, 1.05, 1.25 GB)."""
    got = {w: l2_model.dram_bytes(32, 32, 128, 76, swizzle=w) / 1e9 for w in (4, 8, 16)}
    assert got[8] < got[4] and got[8] < got[16]          # width 8 the least, as measured
    for w, measured in ((4, 1.34), (8, 1.05), (16, 1.25)):
        assert abs(got[w] - measured) / measured < 0.1, (w, got[w], measured)


@pytest.mark.parametrize("M,N,K", [
    (8192, 8192, 8192),      # 75 MB of strips a wave
    (8192, 8192, 7168),      # 66 MB
    (8192, 8192, 5120),      # 47 MB
    (8192, 8192, 4096),      # 38 MB
])
def test_plan_alternates_where_the_model_gains(M, N, K):
    pl = g.plan(M, N, K, max_clusters=76, options=g.Options(cta_group=2, schedule=1))
    mt, nt, kb, G = pl["m_tiles"], pl["n_tiles"], pl["k_blocks"], pl["clusters"]
    up = l2_model.dram_bytes(mt, nt, kb, G)
    alt = l2_model.dram_bytes(mt, nt, kb, G, alternate=True)
    if pl["k_order"] == 1:
        assert alt < 0.85 * up, (up, alt)
    else:
        assert alt > 0.97 * up, (up, alt)
