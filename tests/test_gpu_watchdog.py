"""The device watchdog: a pipeline wait that cannot finish ends the kernel with
a status the host can read, and the context stays usable.

The stall is made with the documented test hook (`inject_stall`): the TMA
producers issue no copies, so the MMA issuer's wait for a filled stage and the
epilogue's wait for an accumulator run into a short limit.  Nothing is copied or
computed, no memory is touched out of bounds, and every wait is bounded.
"""
import numpy as np
import pytest

import oracle
from dense_fp16_gemm_gb300 import inputs
from tests.gpu_util import empty_out, lib_for, to_device, to_host
from tests.tolerance import check_close

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import dense_fp16_gemm_gb300 as g  # noqa: E402


@pytest.mark.parametrize("cg,cp", [(2, 1), (1, 1), (2, 2)])
def test_stalled_pipeline_reports_timeout_then_recovers(cg, cp):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = lib_for(cp)                 # two pairs per cluster: the single-GPU multicast build
    assert g.device_status(lib=lib) == 0
    M, N, K = 512, 512, 256
    A = inputs.draw((M, K), inputs.U, 81)
    B = inputs.draw((N, K), inputs.U, 82)
    Ad, Bd = to_device(A), to_device(B)
    Cd, _ = empty_out(M, N)
    g.gemm_f16_nt(Ad, Bd, Cd, options=g.Options(cta_group=cg, cluster_pairs=cp, inject_stall=1,
                                                timeout_ns=20_000_000), lib=lib)
    word = g.device_status(lib=lib)
    assert word & 1, f"watchdog word {word:#x}"
    sites = {s for s in range(1, 7) if word & (1 << (7 + s))}
    # the MMA issuer (filled slot) and/or the epilogue (finished accumulator) gave up
    assert sites and sites <= {2, 4}, f"unexpected wait sites in {word:#x}"
    assert np.isnan(to_host(Cd).astype(np.float32)).all(), "C was written by a stalled kernel"
    # the context is intact: a normal call right after is correct
    g.gemm_f16_nt(Ad, Bd, Cd, options=g.Options(cta_group=cg, cluster_pairs=cp), lib=lib)
    torch.cuda.synchronize()
    assert g.device_status(lib=lib) == 0
    check_close(to_host(Cd), oracle.gemm_f16_nt(A, B), K, "after watchdog")


def test_deep_k_finishes_inside_the_item_scaled_limit():
    """K = 2^30 with M = N = 8, whole tiles: one 256x256 tile of 2^24 k-blocks on
    one CTA pair, about 4.5 s of tensor work.  The epilogue's wait for the
    accumulator, the MMA issuer's wait for a drained one and the producer's
    waits behind it last the whole item, far beyond the 1 s base limit; their
    limit grows with the tile's k-blocks, so the kernel finishes with the
    watchdog word at 0.  Inputs in {-1, 0, 1}: every partial sum is an integer
    far below 2^24, so the result is exact and must equal the oracle bit for bit
    at the sampled points."""
    M, N, K = 8, 8, 1 << 30
    dev = torch.device("cuda:0")
    free = torch.cuda.mem_get_info(dev)[0]
    if free < 40 * 2**30:
        pytest.skip("needs 32 GiB of free device memory for the operands")
    whole = g.Options(schedule=1)
    pl = g.launch_plan(M, N, K, options=whole)
    assert (pl["num_tiles"], pl["k_blocks"], pl["sk_tiles"], pl["split_pieces"], pl["clusters"]) == \
        (1, 1 << 24, 0, 1, 1)
    Ad = inputs.draw_device_ints((M, K), -1, 1, 2001, dev)
    Bd = inputs.draw_device_ints((N, K), -1, 1, 2002, dev)
    Cd, _ = empty_out(M, N)
    g.gemm_f16_nt(Ad, Bd, Cd, options=whole)
    assert g.device_status() == 0, "a wait ran into the watchdog"
    C = to_host(Cd)
    rows, cols = np.array([0, 7]), np.array([0, 5])
    A_h = Ad[rows].cpu().numpy()
    B_h = Bd[cols].cpu().numpy()
    del Ad, Bd
    torch.cuda.empty_cache()
    rr, cc = np.meshgrid(np.arange(2), np.arange(2), indexing="ij")
    ref, s64 = oracle.gemm_f16_nt_points(A_h, B_h, rr.ravel(), cc.ravel())
    assert np.all(np.abs(s64) < 2 ** 24)
    from tests.tolerance import check_bitexact
    check_bitexact(C[np.ix_(rows, cols)].ravel(), ref, "K = 2^30")
