"""Pins for the CPU oracle, each against something other than the oracle itself.

The oracle computes C_ref[m,n] = RNE_fp16(sum_k A[m,k]·B[n,k]) with an fp64
sequential sum (Tilus matmul-hopper tutorial, "3. Warp Specialization",
§The Full Kernel: A is [m,k], B is [n,k] and the MMA reads B transposed; the
final cast to float16).  Each test below would fail for a plausible mistake:

  * decoding / rounding      -> numpy's own binary16 conversions, all patterns,
                                every tie, and closed-form IEEE-754 cases;
  * transposed operand,      -> identity and a non-involutive permutation;
    wrong index or sign
  * dropped or extra term    -> all-ones closed form RNE16(K) and identity;
  * rounding more than once  -> the sticky-bit case 1 + 2^-11 + 2^-40, whose
    or accumulating in fp32     single rounding differs from any fp32 sum;
  * anything else            -> exact rational arithmetic on every tiny shape,
                                and an exact int64 product for small integers.
"""
from fractions import Fraction

import numpy as np
import pytest

from dense_fp16_gemm_gb300 import inputs

# ---------------------------------------------------------------------------
# helpers written for the tests only
# ---------------------------------------------------------------------------

_ALL = np.arange(65536, dtype=np.uint32).astype(np.uint16)


def _finite_grid():
    """All finite fp16 values as sorted (float64 value, bit pattern) arrays,
    one entry per value (-0 dropped)."""
    h = _ALL.view(np.float16)
    with np.errstate(invalid="ignore"):
        v = h.astype(np.float64)
    ok = np.isfinite(v) & ~((_ALL == 0x8000))
    vals, bits = v[ok], _ALL[ok]
    order = np.argsort(vals, kind="stable")
    return vals[order], bits[order]


_GRID_VALS, _GRID_BITS = _finite_grid()
_MAXF16 = Fraction(65504)


def exact_rne16(q: Fraction) -> int:
    """Round an exact rational to fp16 by searching the enumerated fp16 grid:
    the nearest grid value, ties to the one with an even bit pattern; beyond
    65504 + 16 (half a spacing past the largest value) the result is inf."""
    if q == 0:
        return 0
    if abs(q) >= _MAXF16 + 16:
        return 0xFC00 if q < 0 else 0x7C00
    # bracket q on the grid (float64 values of fp16 are exact fractions)
    i = int(np.searchsorted(_GRID_VALS, float(q)))
    best = None
    for j in range(max(i - 2, 0), min(i + 3, len(_GRID_VALS))):
        d = abs(Fraction(_GRID_VALS[j]) - q)
        key = (d, int(_GRID_BITS[j]) & 1)   # smaller distance, then even significand
        if best is None or key < best[0]:
            best = (key, int(_GRID_BITS[j]))
    return best[1]


def bits(x):
    return np.asarray(x).view(np.uint16)


# ---------------------------------------------------------------------------
# binary16 conversions
# ---------------------------------------------------------------------------

def test_decode_all_patterns_match_numpy(oracle_mod):
    ours = oracle_mod.widen_f16_to_f64(_ALL)
    ref = _ALL.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_round_matches_numpy_on_grid_ties_and_random(oracle_mod):
    g = _GRID_VALS
    mids = (g[:-1] + g[1:]) / 2.0                       # every exact tie
    tests = [g, mids, np.nextafter(mids, np.inf), np.nextafter(mids, -np.inf),
             np.array([65504.0, 65519.999, 65520.0, 65536.0, 1e6, np.inf, -np.inf,
                       2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -25, 2.0 ** -26, 1e-300, -0.0, 0.0])]
    rng = np.random.default_rng(123)
    tests.append(rng.uniform(-70000, 70000, 200000))
    tests.append(rng.uniform(-1, 1, 200000) * 2.0 ** rng.integers(-30, 17, 200000))
    x = np.concatenate(tests)
    ours = bits(oracle_mod.round_f64_to_f16(x))
    with np.errstate(over="ignore"):
        ref = bits(x.astype(np.float16))
    bad = np.flatnonzero(ours != ref)
    assert bad.size == 0, f"{bad.size} mismatches, e.g. x={x[bad[0]]!r} ours={ours[bad[0]]:#x} numpy={ref[bad[0]]:#x}"


@pytest.mark.parametrize("x,expect", [
    (65504.0, 0x7BFF),              # largest finite
    (65519.0, 0x7BFF),              # below the halfway point 65520
    (65520.0, 0x7C00),              # halfway to 65536: ties-to-even overflows to inf
    (-65520.0, 0xFC00),
    (2.0 ** -24, 0x0001),           # smallest subnormal
    (2.0 ** -25, 0x0000),           # halfway between 0 and 2^-24: even is 0
    (3 * 2.0 ** -25, 0x0002),       # halfway between 1 and 2 subnormal ulps: even is 2
    (2.0 ** -14, 0x0400),           # smallest normal
    (2049.0, 0x6800),               # halfway 2048/2050 -> 2048 (even significand)
    (2051.0, 0x6802),               # halfway 2050/2052 -> 2052
    (1.0 + 2.0 ** -11, 0x3C00),     # halfway 1/1+2^-10 -> 1
    (1.0 + 2.0 ** -11 + 2.0 ** -40, 0x3C01),  # just above halfway -> up
    (-0.0, 0x8000),
    (0.0, 0x0000),
])
def test_round_closed_forms(oracle_mod, x, expect):
    assert int(bits(oracle_mod.round_f64_to_f16(np.array([x])))[0]) == expect


# ---------------------------------------------------------------------------
# the product
# ---------------------------------------------------------------------------

def test_identity_returns_A(oracle_mod):
    A = inputs.draw((37, 64), inputs.U, 101)
    B = np.eye(64, dtype=np.float16)
    C = oracle_mod.gemm_f16_nt(A, B)
    assert np.array_equal(bits(C), bits(A))


def test_permutation_pins_transpose(oracle_mod):
    K = 50
    rng = np.random.default_rng(5)
    while True:
        pi = rng.permutation(K)
        if not np.array_equal(pi[pi], np.arange(K)):     # not an involution
            break
    A = inputs.draw((19, K), inputs.U, 102)
    B = np.zeros((K, K), dtype=np.float16)
    B[np.arange(K), pi] = 1.0                            # B[n, pi(n)] = 1
    C = oracle_mod.gemm_f16_nt(A, B)
    assert np.array_equal(bits(C), bits(A[:, pi]))       # C[m,n] = A[m, pi(n)]
    # A·B (no transpose) would give A[:, pi^-1] instead
    assert not np.array_equal(bits(C), bits(A[:, np.argsort(pi)]))


def test_negation_sign(oracle_mod):
    A = inputs.draw((8, 16), inputs.U, 103)
    B = -np.eye(16, dtype=np.float16)
    C = oracle_mod.gemm_f16_nt(A, B)
    assert np.array_equal(C.astype(np.float64), -A.astype(np.float64))


def test_k1_outer_product_single_rounding(oracle_mod):
    a = inputs.draw((200, 1), ("uniform", -300.0, 300.0), 104)
    b = inputs.draw((150, 1), ("uniform", -300.0, 300.0), 105)
    C = oracle_mod.gemm_f16_nt(a, b)
    exact = a.astype(np.float64) * b.astype(np.float64).T   # exact: 11+11 bits
    with np.errstate(over="ignore"):
        assert np.array_equal(bits(C), bits(exact.astype(np.float16)))
    assert np.isinf(C.astype(np.float64)).any()              # some products overflow fp16


@pytest.mark.parametrize("M,N,K", [(64, 48, 5000), (33, 17, 1), (5, 7, 20000)])
def test_small_integers_exact(oracle_mod, M, N, K):
    A = inputs.draw((M, K), inputs.I2, 106 + K)
    B = inputs.draw((N, K), inputs.I2, 107 + K)
    C = oracle_mod.gemm_f16_nt(A, B)
    exact = A.astype(np.int64) @ B.astype(np.int64).T        # exact integer product
    ref = exact.astype(np.float64).astype(np.float16)        # one rounding of an exact integer
    assert np.array_equal(bits(C), bits(ref))


def test_exact_rationals_every_tiny_shape(oracle_mod):
    rng = np.random.default_rng(7)
    shapes = [(m, n, k) for m in range(1, 7) for n in range(1, 7) for k in range(1, 7)]
    shapes += [tuple(int(v) for v in rng.integers(1, 25, 3)) for _ in range(6)]
    for i, (M, N, K) in enumerate(shapes):
        A = inputs.draw((M, K), inputs.U, 1000 + i)
        B = inputs.draw((N, K), ("uniform", -4.0, 4.0), 5000 + i)
        C = oracle_mod.gemm_f16_nt(A, B, threads=1)
        Af = [[Fraction(float(v)) for v in row] for row in A.astype(np.float64)]
        Bf = [[Fraction(float(v)) for v in row] for row in B.astype(np.float64)]
        for m in range(M):
            for n in range(N):
                q = sum(Af[m][k] * Bf[n][k] for k in range(K))
                e = exact_rne16(q)
                got = int(bits(C)[m, n])
                if got != e and not (got in (0, 0x8000) and e in (0, 0x8000)):
                    raise AssertionError(f"shape {(M, N, K)} at {(m, n)}: oracle {got:#x} exact {e:#x}")


@pytest.mark.parametrize("K,expect", [
    (1, 0x3C00), (3, 0x4200), (2047, 0x67FF), (2048, 0x6800), (2049, 0x6800),
    (2051, 0x6802), (4097, 0x6C00), (4098, 0x6C00), (4099, 0x6C01), (65504, 0x7BFF),
    (65519, 0x7BFF), (65520, 0x7C00), (70000, 0x7C00),
])
def test_all_ones_closed_form(oracle_mod, K, expect):
    A = np.ones((2, K), dtype=np.float16)
    B = np.ones((3, K), dtype=np.float16)
    C = oracle_mod.gemm_f16_nt(A, B)
    assert np.all(bits(C) == expect), (K, bits(C))


def test_sticky_bit_single_rounding(oracle_mod):
    # exact sum 1 + 2^-11 + 2^-40 lies just above the fp16 tie between 1 and
    # 1 + 2^-10; an fp32 accumulator loses the 2^-40 and rounds to 1.
    for perm in ([0, 1, 2], [2, 0, 1], [1, 2, 0]):
        a = np.array([[1.0, 2.0 ** -11, 2.0 ** -20]], dtype=np.float16)[:, perm]
        b = np.array([[1.0, 1.0, 2.0 ** -20]], dtype=np.float16)[:, perm]
        assert int(bits(oracle_mod.gemm_f16_nt(a, b))[0, 0]) == 0x3C01


def test_empty_sum_is_positive_zero(oracle_mod):
    A = np.zeros((4, 0), dtype=np.float16)
    B = np.zeros((5, 0), dtype=np.float16)
    C = np.full((4, 5), np.nan, dtype=np.float16)
    oracle_mod.gemm_f16_nt(A, B, C)
    assert np.all(bits(C) == 0)


def test_leading_dimensions_and_untouched_padding(oracle_mod):
    M, N, K = 23, 31, 77
    A = inputs.draw((M, K), inputs.U, 110, ld=K + 9)      # NaN in the padding
    B = inputs.draw((N, K), inputs.U, 111, ld=K + 3)
    Cbuf = np.full((M, N + 5), np.float16(7.0), dtype=np.float16)
    oracle_mod.gemm_f16_nt(A, B, Cbuf[:, :N])
    ref = oracle_mod.gemm_f16_nt(np.ascontiguousarray(A), np.ascontiguousarray(B))
    assert np.array_equal(bits(Cbuf[:, :N]), bits(ref))
    assert np.all(Cbuf[:, N:] == np.float16(7.0))


def test_linearity_on_integers(oracle_mod):
    A = inputs.draw((20, 300), inputs.I2, 112)
    B1 = inputs.draw((30, 300), inputs.I2, 113)
    B2 = inputs.draw((30, 300), inputs.I2, 114)
    S = oracle_mod.gemm_f16_nt_f64
    lhs = S(A, (B1.astype(np.float32) + B2.astype(np.float32)).astype(np.float16))
    assert np.array_equal(lhs, S(A, B1) + S(A, B2))


def test_thread_count_and_points_agree(oracle_mod):
    A = inputs.draw((61, 130), inputs.U, 115)
    B = inputs.draw((45, 130), inputs.U, 116)
    C1 = oracle_mod.gemm_f16_nt(A, B, threads=1)
    C7 = oracle_mod.gemm_f16_nt(A, B, threads=7)
    assert np.array_equal(bits(C1), bits(C7))
    rows = np.array([0, 60, 13, 60, 5])
    cols = np.array([0, 44, 7, 0, 44])
    v, v64 = oracle_mod.gemm_f16_nt_points(A, B, rows, cols)
    assert np.array_equal(bits(v), bits(C1[rows, cols]))
    S = oracle_mod.gemm_f16_nt_f64(A, B)
    assert np.array_equal(v64, S[rows, cols])


def test_output_rounding_error_scale_matches_pages(oracle_mod):
    """With unit-variance outputs at K = 8192, the tutorial quotes a mean
    absolute error of 0.00014 for fp32 accumulation ("6. Register
    Reallocation, Multicast, and a Persistent Kernel", §Shared-Memory Epilogue,
    the Note on fp16 accumulation).  That is the size of the final fp16
    rounding alone, so the oracle's mean |C_ref - S| must sit near it.
    A rounding to bf16, or none at all, would be far off."""
    K = 8192
    s = K ** -0.25
    A = inputs.draw((96, K), ("normal", 0.0, s), 117)
    B = inputs.draw((96, K), ("normal", 0.0, s), 118)
    S = oracle_mod.gemm_f16_nt_f64(A, B)
    C = oracle_mod.gemm_f16_nt(A, B).astype(np.float64)
    assert 0.7 < S.std() < 1.3
    mae = np.abs(C - S).mean()
    assert 1.0e-4 < mae < 1.8e-4, mae
    assert abs(mae - 1.4e-4) < 0.3e-4, mae
