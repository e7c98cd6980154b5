"""Pins for the oracle's bfloat16 variant (bf16 operands and result, fp64 sum,
one round-to-nearest-even to bf16), each against something other than the
oracle itself:

  * decoding            -> numpy's float32 view of the bits shifted up by 16;
  * rounding            -> an exact nearest-value search over the enumerated bf16
                           grid (every value, every tie, neighbours of ties,
                           random doubles) and closed-form IEEE cases;
  * transposition, sign -> identity, non-involutive permutation, negation;
  * the sum             -> exact int64 products of small integers, the all-ones
                           closed form RNE_bf16(K), and a sticky-bit case whose
                           single rounding differs from any fp32 accumulation.
"""
import numpy as np
import pytest

from dense_fp16_gemm_gb300 import inputs

_ALL = np.arange(65536, dtype=np.uint32)


def _grid():
    """All finite bf16 values (from numpy's float32 view), sorted, -0 dropped."""
    with np.errstate(invalid="ignore"):
        v = (_ALL << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    ok = np.isfinite(v) & (_ALL != 0x8000)
    vals, bits = v[ok], _ALL[ok].astype(np.uint16)
    order = np.argsort(vals, kind="stable")
    return vals[order], bits[order]


_VALS, _BITS = _grid()
_MAX = float(_VALS[-1])
_HALF_TOP = 2.0 ** 119          # half the spacing at the top binade (2^127 · 2^-7 / 2)


def exact_rne_bf16(x: np.ndarray) -> np.ndarray:
    """Nearest bf16 by search over the grid, ties to the even bit pattern;
    |x| >= max + half a spacing gives inf.  Differences of adjacent grid
    neighbours are exact in fp64, so every comparison is exact."""
    x = np.asarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    i = np.clip(np.searchsorted(_VALS, x), 1, len(_VALS) - 1)
    lo, hi = _VALS[i - 1], _VALS[i]
    dlo, dhi = x - lo, hi - x
    pick_hi = (dhi < dlo) | ((dhi == dlo) & ((_BITS[i] & 1) == 0))
    out[:] = np.where(pick_hi, _BITS[i], _BITS[i - 1])
    out[(out == 0) & np.signbit(x)] = 0x8000         # negative values that round to zero give -0
    out[x >= _MAX + _HALF_TOP] = 0x7F80
    out[x <= -(_MAX + _HALF_TOP)] = 0xFF80
    return out


def test_decode_all_patterns_match_numpy(oracle_mod):
    ours = oracle_mod.widen_bf16_to_f64(_ALL.astype(np.uint16))
    ref = (_ALL << 16).astype(np.uint32).view(np.float32).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_round_matches_exact_grid_search(oracle_mod):
    g = _VALS
    mids = (g[:-1] + g[1:]) / 2.0
    rng = np.random.default_rng(11)
    x = np.concatenate([g, mids, np.nextafter(mids, np.inf), np.nextafter(mids, -np.inf),
                        rng.uniform(-1, 1, 300000) * 2.0 ** rng.integers(-140, 128, 300000),
                        np.array([_MAX, -_MAX, _MAX + _HALF_TOP, np.nextafter(_MAX + _HALF_TOP, 0),
                                  2.0 ** -133, 2.0 ** -134, 3 * 2.0 ** -134, 1e-300])])
    ours = oracle_mod.round_f64_to_bf16(x)
    ref = exact_rne_bf16(x)
    bad = np.flatnonzero(ours != ref)
    assert bad.size == 0, f"{bad.size} mismatches, e.g. x={x[bad[0]]!r} ours={ours[bad[0]]:#x} exact={ref[bad[0]]:#x}"


@pytest.mark.parametrize("x,expect", [
    (1.0, 0x3F80),
    (1.0 + 2.0 ** -8, 0x3F80),              # halfway 1 / 1+2^-7 -> 1 (even)
    (1.0 + 2.0 ** -8 + 2.0 ** -40, 0x3F81),  # just above halfway -> up
    (257.0, 0x4380),                        # halfway 256 / 258 -> 256
    (259.0, 0x4382),                        # halfway 258 / 260 -> 260
    (2.0 ** -133, 0x0001),                  # smallest subnormal
    (2.0 ** -134, 0x0000),                  # halfway 0 / 2^-133 -> 0
    (3 * 2.0 ** -134, 0x0002),              # halfway 1 / 2 ulps -> 2
    (2.0 ** -126, 0x0080),                  # smallest normal
    (-0.0, 0x8000),
    (3.3895313892515355e38, 0x7F7F),        # largest finite
    (3.3961775292304986e38, 0x7F80),        # halfway to 2^128: overflow
])
def test_round_closed_forms(oracle_mod, x, expect):
    assert int(oracle_mod.round_f64_to_bf16(np.array([x]))[0]) == expect


def _f(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_identity_permutation_and_sign(oracle_mod):
    K = 48
    A = inputs.draw_bf16((21, K), inputs.U, 201)
    eye = exact_rne_bf16(np.eye(K))
    assert np.array_equal(oracle_mod.gemm_bf16_nt(A, eye), A)
    rng = np.random.default_rng(3)
    while True:
        pi = rng.permutation(K)
        if not np.array_equal(pi[pi], np.arange(K)):
            break
    P = np.zeros((K, K), dtype=np.uint16)
    P[np.arange(K), pi] = 0x3F80                     # 1.0
    assert np.array_equal(oracle_mod.gemm_bf16_nt(A, P), A[:, pi])
    assert not np.array_equal(oracle_mod.gemm_bf16_nt(A, P), A[:, np.argsort(pi)])
    neg_eye = (eye | np.where(eye != 0, 0x8000, 0)).astype(np.uint16)      # -I
    neg_a = (A ^ np.where(A != 0, 0x8000, 0)).astype(np.uint16)
    assert np.array_equal(oracle_mod.gemm_bf16_nt(A, neg_eye), neg_a)


def test_k1_outer_product(oracle_mod):
    a = inputs.draw_bf16((120, 1), ("uniform", -1e20, 1e20), 202)
    b = inputs.draw_bf16((90, 1), ("uniform", -1e20, 1e20), 203)
    C = oracle_mod.gemm_bf16_nt(a, b)
    exact = _f(a) * _f(b).T                          # 8 + 8 significant bits: exact
    assert np.array_equal(C, exact_rne_bf16(exact))
    assert (C == 0x7F80).any() or (C == 0xFF80).any()   # some products overflow


@pytest.mark.parametrize("M,N,K", [(40, 30, 3000), (9, 11, 1)])
def test_small_integers_exact(oracle_mod, M, N, K):
    A = inputs.draw_bf16((M, K), inputs.I2, 204 + K)
    B = inputs.draw_bf16((N, K), inputs.I2, 205 + K)
    exact = _f(A).astype(np.int64) @ _f(B).astype(np.int64).T
    assert np.array_equal(oracle_mod.gemm_bf16_nt(A, B), exact_rne_bf16(exact.astype(np.float64)))


@pytest.mark.parametrize("K,expect", [(1, 0x3F80), (255, 0x437F), (256, 0x4380), (257, 0x4380),
                                      (259, 0x4382), (513, 0x4400), (514, 0x4400),
                                      (515, 0x4401), (518, 0x4402)])
def test_all_ones_closed_form(oracle_mod, K, expect):
    A = np.full((2, K), 0x3F80, dtype=np.uint16)
    B = np.full((3, K), 0x3F80, dtype=np.uint16)
    assert np.all(oracle_mod.gemm_bf16_nt(A, B) == expect)


def test_sticky_bit_single_rounding(oracle_mod):
    # 1 + 2^-8 + 2^-40: just above the bf16 tie between 1 and 1 + 2^-7
    one, t8, t20 = 0x3F80, 0x3B80, 0x3580            # 1, 2^-8, 2^-20
    for perm in ([0, 1, 2], [2, 0, 1]):
        a = np.array([[one, t8, t20]], dtype=np.uint16)[:, perm]
        b = np.array([[one, one, t20]], dtype=np.uint16)[:, perm]
        assert int(oracle_mod.gemm_bf16_nt(a, b)[0, 0]) == 0x3F81


def test_points_match_full(oracle_mod):
    A = inputs.draw_bf16((33, 70), inputs.U, 206)
    B = inputs.draw_bf16((17, 70), inputs.U, 207)
    C = oracle_mod.gemm_bf16_nt(A, B)
    rows, cols = np.array([0, 32, 5]), np.array([16, 0, 7])
    assert np.array_equal(oracle_mod.gemm_bf16_nt_points(A, B, rows, cols), C[rows, cols])
