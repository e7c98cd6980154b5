"""Pins for the oracle's fp16-accumulation variant (the accumulator rounded to
fp16 after every 16-wide k step), each against something other than the
oracle itself:

  * one step            -> for K <= 16 the recurrence is one rounding of the
                           exact sum: the fp32-accumulation oracle's result;
  * the recurrence      -> closed forms: all-ones sums grow by 16 per step and
                           stall at 32768, where adding 16 is a tie that rounds
                           back to the even value; constructed sums whose
                           per-step roundings lose what one final rounding
                           keeps, placed so that a step of 8 or 32 gives a
                           different answer than a step of 16;
  * sign, overflow      -> negating A negates C; a step past 65520 gives inf
                           and the accumulator stays there;
  * the pages' numbers  -> over a K = 8192 reduction with unit-variance outputs
                           the mean absolute error against the exact sum is
                           0.0023 with fp16 accumulation and 0.00014 with fp32
                           ("6. Register Reallocation, Multicast, and a
                           Persistent Kernel", §Shared-Memory Epilogue, the Note
                           on an earlier fp16-accumulating version); the
                           maximum there was 0.047.
"""
import numpy as np
import pytest

from dense_fp16_gemm_gb300 import inputs


@pytest.mark.parametrize("K", [1, 5, 16])
def test_single_step_is_one_rounding(oracle_mod, K):
    A = inputs.draw((37, K), inputs.U, 300 + K)
    B = inputs.draw((29, K), inputs.U, 301 + K)
    assert np.array_equal(oracle_mod.gemm_f16_nt_acc16(A, B).view(np.uint16),
                          oracle_mod.gemm_f16_nt(A, B).view(np.uint16))


@pytest.mark.parametrize("K,expect", [(16, 16.0), (2048, 2048.0), (20000, 20000.0), (32768, 32768.0),
                                      (32784, 32768.0), (40000, 32768.0), (20008, 20000.0)])
def test_all_ones_grow_by_16_and_stall(oracle_mod, K, expect):
    # each step adds 16: exact while the grid spacing is <= 16 (below 32768);
    # at 32768 the spacing is 32, 32768 + 16 is a tie and rounds to the even 32768.
    # K = 20008: the last, 8-wide step gives 20008, which rounds to 20000 (spacing 16).
    one_a = np.ones((2, K), dtype=np.float16)
    one_b = np.ones((3, K), dtype=np.float16)
    C = oracle_mod.gemm_f16_nt_acc16(one_a, one_b).astype(np.float64)
    assert np.all(C == expect)


def _sparse_row(K, entries):
    r = np.zeros(K, dtype=np.float16)
    for k, v in entries.items():
        r[k] = v
    return r[None, :]


def test_per_step_rounding_loses_what_one_rounding_keeps(oracle_mod):
    # step 0 sums to 2049 -> 2048 (tie, even); step 1 adds 1: 2049 -> 2048.
    # One final rounding of the exact 2050 gives 2050.
    K = 32
    a = _sparse_row(K, {0: 2048.0, 1: 1.0, 16: 1.0})
    b = np.ones((1, K), dtype=np.float16)
    assert float(oracle_mod.gemm_f16_nt_acc16(a, b)[0, 0]) == 2048.0
    assert float(oracle_mod.gemm_f16_nt(a, b)[0, 0]) == 2050.0


def test_step_is_sixteen_wide(oracle_mod):
    # 2048 + 1 at k = 0, 1 and 1 more at k = 8: one 16-wide step holds 2050 exactly;
    # 8-wide steps would round 2049 -> 2048 first and end at 2048 (2049 -> 2048 again).
    K = 16
    a = _sparse_row(K, {0: 2048.0, 1: 1.0, 8: 1.0})
    b = np.ones((1, K), dtype=np.float16)
    assert float(oracle_mod.gemm_f16_nt_acc16(a, b)[0, 0]) == 2050.0
    # and the step boundary sits at k = 16, not 32: 2048 + 1 at k = 15, then 1 at k = 16
    K = 32
    a = _sparse_row(K, {0: 2048.0, 15: 1.0, 16: 1.0})
    b = np.ones((1, K), dtype=np.float16)
    assert float(oracle_mod.gemm_f16_nt_acc16(a, b)[0, 0]) == 2048.0


def test_negation_and_overflow(oracle_mod):
    A = inputs.draw((21, 300), inputs.U, 311)
    B = inputs.draw((17, 300), inputs.U, 312)
    C = oracle_mod.gemm_f16_nt_acc16(A, B).astype(np.float64)
    Cn = oracle_mod.gemm_f16_nt_acc16(-A, B).astype(np.float64)
    assert np.array_equal(Cn, -C)
    # 16 products of 2048·16 = 524288 > 65520: inf after the first step, and it stays
    a = np.full((1, 48), 2048.0, dtype=np.float16)
    b = np.concatenate([np.full(16, 16.0), np.full(32, -1.0)]).astype(np.float16)[None, :]
    assert np.isposinf(float(oracle_mod.gemm_f16_nt_acc16(a, b)[0, 0]))


def test_error_statistics_match_the_pages(oracle_mod):
    K = 8192
    sig = K ** -0.25                      # unit-variance outputs: K·sig⁴ = 1
    rng = np.random.default_rng(8192)
    A = (rng.standard_normal((48, K)) * sig).astype(np.float16)
    B = (rng.standard_normal((48, K)) * sig).astype(np.float16)
    exact = oracle_mod.gemm_f16_nt_f64(A, B)
    assert 0.9 < exact.std() < 1.1
    err16 = np.abs(oracle_mod.gemm_f16_nt_acc16(A, B).astype(np.float64) - exact)
    err32 = np.abs(oracle_mod.gemm_f16_nt(A, B).astype(np.float64) - exact)
    assert 0.0018 < err16.mean() < 0.0029, err16.mean()       # pages: 0.0023
    assert 0.00011 < err32.mean() < 0.00017, err32.mean()     # pages: 0.00014
    assert err16.max() <= 0.047                               # pages' maximum, over far more outputs


def test_points_match_full(oracle_mod):
    A = inputs.draw((33, 200), inputs.U, 313)
    B = inputs.draw((17, 200), inputs.U, 314)
    C = oracle_mod.gemm_f16_nt_acc16(A, B)
    rows, cols = np.array([0, 32, 5]), np.array([16, 0, 7])
    assert np.array_equal(oracle_mod.gemm_f16_nt_acc16_points(A, B, rows, cols).view(np.uint16),
                          C[rows, cols].view(np.uint16))
