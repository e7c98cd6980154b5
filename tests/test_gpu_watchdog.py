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
from tests.gpu_util import empty_out, to_device, to_host
from tests.tolerance import check_close

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import dense_fp16_gemm_gb300 as g  # noqa: E402


@pytest.mark.parametrize("cg,cp", [(2, 1), (1, 1), (2, 2)])
def test_stalled_pipeline_reports_timeout_then_recovers(cg, cp):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    assert g.device_status() == 0
    M, N, K = 512, 512, 256
    A = inputs.draw((M, K), inputs.U, 81)
    B = inputs.draw((N, K), inputs.U, 82)
    Ad, Bd = to_device(A), to_device(B)
    Cd, _ = empty_out(M, N)
    g.gemm_f16_nt(Ad, Bd, Cd, options=g.Options(cta_group=cg, cluster_pairs=cp, inject_stall=1,
                                                timeout_ns=20_000_000))
    word = g.device_status()
    assert word & 1, f"watchdog word {word:#x}"
    sites = {s for s in range(1, 7) if word & (1 << (7 + s))}
    # the MMA issuer (filled slot) and/or the epilogue (finished accumulator) gave up
    assert sites and sites <= {2, 4}, f"unexpected wait sites in {word:#x}"
    assert np.isnan(to_host(Cd).astype(np.float32)).all(), "C was written by a stalled kernel"
    # the context is intact: a normal call right after is correct
    g.gemm_f16_nt(Ad, Bd, Cd, options=g.Options(cta_group=cg, cluster_pairs=cp))
    torch.cuda.synchronize()
    assert g.device_status() == 0
    check_close(to_host(Cd), oracle.gemm_f16_nt(A, B), K, "after watchdog")
