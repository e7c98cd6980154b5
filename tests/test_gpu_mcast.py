"""The single-GPU multicast build (libgemm_f16_nt_mcast.so): its tensor maps
may cover only the current GPU's own device memory.  Operands elsewhere
(pinned host memory here) are refused with GEMM_ERR_NOT_LOCAL before anything
is enqueued, so C stays untouched; device operands run two pairs per cluster
and match the oracle.
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

NOT_LOCAL = 7


@pytest.fixture(autouse=True)
def _needs_one_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    if torch.cuda.device_count() != 1:
        pytest.skip("the multicast build runs only in a process that sees one GPU")
    yield
    assert g.device_status(lib=g.library_mcast()) == 0


def _call(lib, A, B, C):
    M, K = A.shape
    N = B.shape[0]
    return lib.gemm_f16_nt(M, N, K, A.data_ptr(), A.stride(0), B.data_ptr(), B.stride(0), C.data_ptr(),
                           C.stride(0), torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("which", ["A", "B", "both"])
def test_host_operands_refused_without_a_launch(which):
    mc = g.library_mcast()
    M, N, K = 1000, 1500, 1000                     # K = 1000: pitch not a multiple of 64, two pairs
    A = inputs.draw((M, K), inputs.U, 3501)
    B = inputs.draw((N, K), inputs.U, 3502)
    Ad, Bd = to_device(A), to_device(B)
    Ah = torch.from_numpy(A).pin_memory()
    Bh = torch.from_numpy(B).pin_memory()
    a = Ah if which in ("A", "both") else Ad
    b = Bh if which in ("B", "both") else Bd
    C, _ = empty_out(M, N)
    torch.cuda.synchronize()
    assert _call(mc, a, b, C) == NOT_LOCAL
    torch.cuda.synchronize()
    assert torch.isnan(C).all().item(), "C was written by a refused call"


def test_device_operands_run_two_pairs():
    mc = g.library_mcast()
    M, N, K = 1000, 1500, 1000
    pl = g.launch_plan(M, N, K, lib=mc)
    assert pl["cluster_pairs"] == 2
    A = inputs.draw((M, K), inputs.U, 3503)
    B = inputs.draw((N, K), inputs.U, 3504)
    C, _ = empty_out(M, N)
    assert _call(mc, to_device(A), to_device(B), C) == 0
    torch.cuda.synchronize()
    check_close(to_host(C), oracle.gemm_f16_nt(A, B), K, "multicast build")
