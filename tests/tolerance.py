"""The parity tolerance between the CUDA path and the oracle.

Per element: |C_gpu - C_ref| <= 2 * ulp16(|C_ref|) + 1e-4 * sqrt(K), where
ulp16(x) = 2^(max(floor(log2 x), -14) - 10) is the spacing of the fp16 grid at
x (2^-24 at zero).  Two ulps cover the GPU's double rounding (fp32 accumulator,
then fp16) plus its fp32 accumulation error; the sqrt(K) term covers outputs
near zero, where the fp32 error of a K-term sum is not small against ulp16.
An infinite reference must be matched exactly and NaN is never accepted.
Integer-valued inputs whose partial sums all stay below 2^24 must match bit
for bit (-0 and +0 compare equal).
"""
import numpy as np


def ulp16(x) -> np.ndarray:
    a = np.abs(np.asarray(x, dtype=np.float64))
    _, e2 = np.frexp(a)                      # a = f * 2^e2, f in [0.5, 1)
    e = np.where(a > 0, np.maximum(e2.astype(np.int64) - 1, -14), -14)
    return np.ldexp(1.0, e - 10)


def ulp_bf16(x) -> np.ndarray:
    """Spacing of the bfloat16 grid at |x| (7 fraction bits, normal from 2^-126)."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    _, e2 = np.frexp(a)
    e = np.where(a > 0, np.maximum(e2.astype(np.int64) - 1, -126), -126)
    return np.ldexp(1.0, e - 7)


def bf16_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64, through numpy's float32 view."""
    b = np.asarray(bits).view(np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def check_close(c_gpu, c_ref, K: int, where: str = "", ulp=None):
    """Assert the per-element tolerance (2 ulps of the output format + 1e-4
    sqrt(K)); returns the worst ratio err/bound.  Arrays may be fp16 values or
    float64 values of another format with its `ulp` function."""
    ulp = ulp or ulp16
    g = np.asarray(c_gpu).astype(np.float64)
    r = np.asarray(c_ref).astype(np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    assert not np.isnan(g).any(), f"{where}: NaN in GPU output at {np.argwhere(np.isnan(g))[:5]}"
    inf_ref = np.isinf(r)
    if inf_ref.any():
        assert np.array_equal(g[inf_ref], r[inf_ref]), f"{where}: inf mismatch"
    fin = ~inf_ref
    assert not np.isinf(g[fin]).any(), f"{where}: GPU inf where the reference is finite"
    bound = 2.0 * ulp(r[fin]) + 1e-4 * np.sqrt(max(K, 1))
    err = np.abs(g[fin] - r[fin])
    ratio = err / bound
    if ratio.size and ratio.max() > 1.0:
        idx = np.argmax(ratio)
        flat = np.flatnonzero(fin.ravel())[idx]
        pos = np.unravel_index(flat, r.shape)
        raise AssertionError(
            f"{where}: |gpu-ref| above tolerance at {pos}: gpu={g[pos]!r} ref={r[pos]!r} "
            f"err={err[idx]:.3e} bound={bound[idx]:.3e}; "
            f"{int((ratio > 1).sum())} elements out of tolerance")
    return float(ratio.max()) if ratio.size else 0.0


def check_bitexact(c_gpu, c_ref, where: str = ""):
    g = np.asarray(c_gpu).view(np.uint16).astype(np.uint32)
    r = np.asarray(c_ref).view(np.uint16).astype(np.uint32)
    # +0 and -0 compare equal
    g = np.where(g == 0x8000, 0, g)
    r = np.where(r == 0x8000, 0, r)
    bad = np.argwhere(g != r)
    assert bad.size == 0, (f"{where}: {len(bad)} elements differ in bits, first at "
                           f"{tuple(bad[0])}: gpu=0x{int(g[tuple(bad[0])]):04x} "
                           f"ref=0x{int(r[tuple(bad[0])]):04x}")
