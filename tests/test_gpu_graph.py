"""The GEMM captured into a CUDA graph and replayed with new inputs.

A shape whose plain call splits tiles in k (stream-K) is captured: the
captured launch must be planned without the split (its completion flags are
tagged per launch, and a replay repeats the launch's parameters), and every
replay must compute the product of the inputs it finds.  Small-integer inputs
keep every sum exact, so the comparison is exact.
"""
import numpy as np
import pytest

from dense_fp16_gemm_gb300 import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import dense_fp16_gemm_gb300 as g  # noqa: E402


@pytest.fixture(autouse=True)
def _needs_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    assert g.device_status() == 0, "watchdog word set after the case"


def _operands(M, N, K, seed):
    A = inputs.draw((M, K), inputs.I2, seed)
    A = (A * (np.arange(K) % 4 == 0)).astype(np.float16)     # sums stay small integers
    B = inputs.draw((N, K), inputs.I2, seed + 1)
    return A, B


@pytest.mark.parametrize("M,N,K", [(1024, 1024, 8192), (256, 256, 8192)])
def test_captured_gemm_replays_with_new_inputs(M, N, K):
    lim = g.device_limits()
    # (cta_group 2: the persistent kernel, whose split in k the capture must turn off)
    pl = g.plan(M, N, K, num_sms=lim["sms"], max_clusters=lim["resident_pairs"], options=g.Options(cta_group=2))
    assert pl["sk_tiles"] > 0 or pl["split_pieces"] > 1     # split in k when called directly
    A0, B0 = _operands(M, N, K, 700)
    As = torch.from_numpy(A0).cuda()
    Bs = torch.from_numpy(B0).cuda()
    Cs = torch.empty((M, N), dtype=torch.float16, device="cuda")
    items = 64
    trace = torch.zeros((lim["resident_pairs"] * items * 8,), dtype=torch.int64, device="cuda")
    opts = g.Options(trace=trace.data_ptr(), trace_items=items, cta_group=2)
    g.gemm_f16_nt(As, Bs, Cs, options=opts)          # warm-up outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        g.gemm_f16_nt(As, Bs, Cs, options=opts)
    for r in range(3):
        A, B = _operands(M, N, K, 710 + 10 * r)
        As.copy_(torch.from_numpy(A))
        Bs.copy_(torch.from_numpy(B))
        trace.zero_()
        graph.replay()
        torch.cuda.synchronize()
        exact = A.astype(np.float64) @ B.astype(np.float64).T
        assert np.abs(exact).max() < 2048
        assert np.array_equal(Cs.cpu().numpy().astype(np.float64), exact), f"replay {r}"
        kinds = (trace.view(-1, items, 8)[:, :, 0].cpu().numpy() >> 32)
        used = trace.view(-1, items, 8)[:, :, 2].cpu().numpy() != 0
        assert used.any() and np.all(kinds[used] == 0), "the captured launch split tiles in k"


def test_captured_gemm_with_a_partial_last_wave():
    """A shape whose last, partial wave is claimed at run time when called
    directly (45 tiles on 7 clusters, 3 left over): the captured launch deals
    it round-robin instead (a replay repeats the launch's tag on the claim
    counter), and every replay computes the product of its inputs."""
    M, N, K = 1100, 2100, 520
    opts = g.Options(cta_group=2, max_clusters=7, schedule=1)
    assert g.plan(M, N, K, options=opts)["claimed_tiles"] == 45 % 7
    A0, B0 = _operands(M, N, K, 800)
    As = torch.from_numpy(A0).cuda()
    Bs = torch.from_numpy(B0).cuda()
    Cs = torch.empty((M, N + (-N) % 8), dtype=torch.float16, device="cuda")[:, :N]
    g.gemm_f16_nt(As, Bs, Cs, options=opts)          # warm-up outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        inside = g.launch_plan(M, N, K, stream=torch.cuda.current_stream(), options=opts)
        g.gemm_f16_nt(As, Bs, Cs, options=opts)
    assert inside["claimed_tiles"] == 0
    for r in range(3):
        A, B = _operands(M, N, K, 810 + 10 * r)
        As.copy_(torch.from_numpy(A))
        Bs.copy_(torch.from_numpy(B))
        graph.replay()
        torch.cuda.synchronize()
        exact = A.astype(np.float64) @ B.astype(np.float64).T
        assert np.abs(exact).max() < 2048
        assert np.array_equal(Cs.cpu().numpy().astype(np.float64), exact), f"replay {r}"
