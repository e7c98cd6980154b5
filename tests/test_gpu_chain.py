"""Back-to-back launches that feed each other on one stream.

Each launch may start its set-up while the launch before it on the stream is
still running (programmatic dependent launch); it must read its operands only
after that launch has finished writing them.  Here every GEMM's A operand is
the previous GEMM's C, with no synchronisation in between:

    X_{t+1} = X_t · Pᵀ,   P[n, k] = 1 if k = π(n) else 0,

so X_{t+1}[m, n] = X_t[m, π(n)] and X_T[m, n] = X_0[m, π^T(n)].  X_0 holds
small integers and P is a permutation matrix, so every step is exact whatever
the summation order: the result must match the composed permutation exactly.
A launch that read a stale or half-written X would break the equality.
"""
import numpy as np
import pytest

from dense_fp16_gemm_gb300 import inputs
from tests.gpu_util import lib_for

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import dense_fp16_gemm_gb300 as g  # noqa: E402


@pytest.fixture(autouse=True)
def _needs_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    assert g.device_status() == 0, "watchdog word set after the case"


def _perm_matrix(pi: np.ndarray, dtype):
    n = len(pi)
    P = torch.zeros((n, n), dtype=dtype)
    P[torch.arange(n), torch.from_numpy(pi)] = 1
    return P


# (M, K = N, schedule, cluster_pairs): whole tiles, stream-K, two pairs with
# A multicast, and a row pitch that is not a multiple of 64 elements
CASES = [(8192, 1024, 1, 1), (2048, 2048, 2, 1), (4096, 1536, 0, 2), (3000, 1000, 0, 0)]


@pytest.mark.parametrize("M,KN,schedule,pairs", CASES)
@pytest.mark.parametrize("bf16", [False, True])
def test_chained_permutations_are_exact(M, KN, schedule, pairs, bf16):
    steps = 16
    rng = np.random.default_rng(1000 + M + KN)
    pi = rng.permutation(KN)
    dt = torch.bfloat16 if bf16 else torch.float16
    x0 = inputs.draw((M, KN), ("int", -8, 8), 77 + KN).astype(np.float32)
    X = [torch.from_numpy(x0).to(dt).cuda(), torch.full((M, KN), float("nan"), dtype=dt, device="cuda")]
    P = _perm_matrix(pi, dt).cuda()
    fn = g.gemm_bf16_nt if bf16 else g.gemm_f16_nt
    o = g.Options(schedule=schedule, cluster_pairs=pairs)
    torch.cuda.synchronize()
    for t in range(steps):
        fn(X[t % 2], P, X[(t + 1) % 2], options=o, lib=lib_for(pairs))
    torch.cuda.synchronize()
    idx = np.arange(KN)
    for _ in range(steps):
        idx = pi[idx]
    expect = x0[:, idx]
    got = X[steps % 2].float().cpu().numpy()
    bad = np.flatnonzero(got != expect)
    assert bad.size == 0, f"{bad.size} elements differ, first at {np.unravel_index(bad[0], got.shape)}"


def test_chain_across_streams_with_events():
    """Two streams, each GEMM waiting on an event recorded after the one before:
    cross-stream order comes from the event, not from stream order."""
    M, KN, steps = 4096, 1024, 8
    rng = np.random.default_rng(5)
    pi = rng.permutation(KN)
    x0 = inputs.draw((M, KN), ("int", -8, 8), 91).astype(np.float32)
    X = [torch.from_numpy(x0).half().cuda(), torch.empty((M, KN), dtype=torch.float16, device="cuda")]
    P = _perm_matrix(pi, torch.float16).cuda()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    torch.cuda.synchronize()
    ev = None
    for t in range(steps):
        s = streams[t % 2]
        if ev is not None:
            s.wait_event(ev)
        g.gemm_f16_nt(X[t % 2], P, X[(t + 1) % 2], stream=s)
        ev = torch.cuda.Event()
        ev.record(s)
    torch.cuda.synchronize()
    idx = np.arange(KN)
    for _ in range(steps):
        idx = pi[idx]
    assert np.array_equal(X[steps % 2].float().cpu().numpy(), x0[:, idx])
