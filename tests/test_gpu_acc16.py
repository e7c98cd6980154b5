"""Parity of the fp16-accumulation variant (options.accumulate = 1) with the
oracle's model of it: the accumulator rounded to fp16 (nearest, ties to even)
after every 16-wide k step, each step's sum exact.

The bar:
  * exact where nothing rounds (small-integer inputs) and on the closed forms
    that pin the rounding itself (all-ones sums stall at 32768; per-step ties
    lose what one final rounding keeps);
  * on random data, at least 98 % of the outputs bit-identical to the model and
    every output within 8 fp16 ulps of the outputs' rms magnitude of it: the
    tensor cores' internal sum of a 16-wide step can differ from the exact one
    in its last place, and a step where that changes the rounding leaves the
    accumulator one ulp apart from then on (measured on GB300: 99.9 % identical
    at K = 64, 99 % at K = 8192);
  * the error against the exact sum has the pages' statistics: mean 0.0023 over
    a K = 8192 reduction with unit-variance outputs (0.00014 with fp32
    accumulation), maximum 0.047 ("6. Register Reallocation, Multicast, and a
    Persistent Kernel", §Shared-Memory Epilogue, the Note).
"""
import numpy as np
import pytest

import oracle
from dense_fp16_gemm_gb300 import inputs
from tests.gpu_util import empty_out, lib_for, to_device, to_host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

import dense_fp16_gemm_gb300 as g  # noqa: E402


@pytest.fixture(autouse=True)
def _needs_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    yield
    assert g.device_status() == 0, "watchdog word set after the case"


def run(A, B, **kw):
    M, N = A.shape[0], B.shape[0]
    Cd, Cbuf = empty_out(M, N)
    g.gemm_f16_nt(to_device(A), to_device(B), Cd, options=g.Options(accumulate=1, **kw),
                  lib=lib_for(kw.get("cluster_pairs", 0)))
    torch.cuda.synchronize()
    assert np.isnan(to_host(Cbuf)[:M, N:].astype(np.float32)).all(), "padding columns of C were written"
    return to_host(Cd)


@pytest.mark.parametrize("M,N,K,cg,cp", [(300, 520, 328, 2, 0), (7, 9, 3, 2, 0), (1000, 700, 1000, 2, 2),
                                         (513, 1025, 200, 1, 0), (256, 256, 4096, 2, 1)])
def test_integer_inputs_exact(M, N, K, cg, cp):
    A = inputs.draw((M, K), inputs.I2, 400 + K)
    B = inputs.draw((N, K), inputs.I2, 401 + K)
    if K > 500:   # keep every partial sum an integer below 2048, exact in fp16
        A = (A * (np.arange(K) % 4 == 0)).astype(np.float16)
    C = run(A, B, cta_group=cg, cluster_pairs=cp)
    exact = A.astype(np.float64) @ B.astype(np.float64).T
    assert np.abs(exact).max() < 2048
    assert np.array_equal(C.astype(np.float64), exact)
    assert np.array_equal(C.view(np.uint16), oracle.gemm_f16_nt_acc16(A, B).view(np.uint16))


@pytest.mark.parametrize("K,expect", [(40000, 32768.0), (32784, 32768.0), (20008, 20000.0), (2048, 2048.0)])
def test_all_ones_stall_like_the_model(K, expect):
    one = np.ones((256, K), dtype=np.float16)
    C = run(one, one[:128])
    assert np.all(C.astype(np.float64) == expect)


@pytest.mark.parametrize("K,entries,expect", [
    (32, {0: 2048.0, 1: 1.0, 16: 1.0}, 2048.0),     # two per-step ties lose 2 (exact 2050)
    (16, {0: 2048.0, 1: 1.0, 8: 1.0}, 2050.0),      # one 16-wide step holds 2050
    (32, {0: 2048.0, 15: 1.0, 16: 1.0}, 2048.0),    # the step boundary is at k = 16
    (16, {0: 1.0, 1: 2.0 ** -11, 2: 2.0 ** -20}, 1.0 + 2.0 ** -10),   # sticky bit past the tie
])
def test_per_step_rounding_like_the_model(K, entries, expect):
    a = np.zeros((256, K), dtype=np.float16)
    for k, v in entries.items():
        a[:, k] = v
    b = np.ones((256, K), dtype=np.float16)
    C = run(a, b)
    assert np.all(C.astype(np.float64) == expect)
    assert float(oracle.gemm_f16_nt_acc16(a[:1], b[:1])[0, 0]) == expect


@pytest.mark.parametrize("M,N,K", [(512, 384, 64), (300, 520, 1000), (512, 512, 8192)])
def test_random_inputs_follow_the_model(M, N, K):
    A = inputs.draw((M, K), inputs.U, 410 + K)
    B = inputs.draw((N, K), inputs.U, 411 + K)
    C = run(A, B).astype(np.float64)
    ref = oracle.gemm_f16_nt_acc16(A, B).astype(np.float64)
    same = np.mean(C == ref)
    rms = np.sqrt(np.mean(ref ** 2))
    ulp_rms = 2.0 ** (np.floor(np.log2(rms)) - 10)
    worst = np.abs(C - ref).max()
    assert same >= 0.98, f"only {same:.4f} of the outputs match the model"
    assert worst <= 8 * ulp_rms, f"max |gpu - model| = {worst} > 8 ulp16({rms:.3g})"


def test_error_statistics_match_the_pages():
    K = 8192
    sig = K ** -0.25                      # unit-variance outputs: K·sig⁴ = 1
    rng = np.random.default_rng(8192)
    A = (rng.standard_normal((512, K)) * sig).astype(np.float16)
    B = (rng.standard_normal((512, K)) * sig).astype(np.float16)
    exact = oracle.gemm_f16_nt_f64(A, B)
    err16 = np.abs(run(A, B).astype(np.float64) - exact)
    Cd, _ = empty_out(512, 512)
    g.gemm_f16_nt(to_device(A), to_device(B), Cd)
    torch.cuda.synchronize()
    err32 = np.abs(to_host(Cd).astype(np.float64) - exact)
    assert 0.0018 < err16.mean() < 0.0029, err16.mean()       # pages: 0.0023
    assert 0.00011 < err32.mean() < 0.00017, err32.mean()     # pages: 0.00014
    assert err16.max() <= 0.047


def test_mn_major_operands():
    M, N, K = 300, 200, 256
    A = inputs.draw((M, K), inputs.I2, 420)
    B = inputs.draw((N, K), inputs.I2, 421)
    Cd, _ = empty_out(M, N)
    g.gemm_f16_nt(to_device(np.ascontiguousarray(A.T)), to_device(np.ascontiguousarray(B.T)), Cd,
                  options=g.Options(accumulate=1), a_layout=1, b_layout=1)
    torch.cuda.synchronize()
    assert np.array_equal(to_host(Cd).astype(np.float64), A.astype(np.float64) @ B.astype(np.float64).T)
