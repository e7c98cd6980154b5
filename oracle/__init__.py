"""CPU oracle for C[M,N] = A[M,K] · B[N,K]ᵀ (fp16 in, fp16 out).

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  The product
library (``dense_fp16_gemm_gb300``) never imports, links or calls it, and this
package never imports the product.

The arithmetic lives in ``gemm_oracle.c`` (plain C, compiled here with gcc
without fast-math and without floating-point contraction); this module only
builds it and marshals numpy arrays.  Every element is a sequential fp64 sum over
k followed by one round-to-nearest-even to fp16 (Tilus matmul-hopper tutorial,
"3. Warp Specialization", §The Full Kernel for the operand layout; the final
``cast(acc, float16)`` for the single rounding).

Functions take and return fp16 data as ``numpy.float16`` arrays (bit patterns
are what matter; they are reinterpreted as uint16 at the C boundary).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gemm_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle_gemm.so")

_lock = threading.Lock()
_default = None

_i64 = ctypes.c_int64
_p = ctypes.c_void_p


def compile_source(src: str, out_path: str) -> str:
    """gcc the given oracle C file into a shared library at out_path."""
    os.makedirs(os.path.dirname(out_path), exist_ok=True)
    tmp = out_path + ".%d.tmp" % os.getpid()
    cmd = ["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-std=c11",
           "-D_GNU_SOURCE", "-fPIC", "-shared", "-Wall", "-o", tmp, src,
           "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out_path)
    return out_path


def build(force: bool = False) -> str:
    """Compile the oracle shared library with gcc; returns its path."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    return compile_source(_SRC, _LIB_PATH)


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover - non-Linux
        return max(1, os.cpu_count() or 1)


def _rows(x: np.ndarray, name: str, dtype=np.float16):
    """(pointer, leading dimension) of a 2-D 16-bit array with unit column stride."""
    if x.dtype != dtype or x.ndim != 2:
        raise TypeError(f"{name} must be a 2-D {np.dtype(dtype).name} array")
    if x.shape[1] > 1 and x.strides[1] != 2:
        raise ValueError(f"{name} must have unit stride along its last axis")
    ld = x.strides[0] // 2 if x.shape[0] > 1 else max(x.shape[1], 1)
    return x.ctypes.data, ld


class Oracle:
    """The oracle functions bound to one compiled copy of gemm_oracle.c."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        lib.oracle_gemm_f16_nt.argtypes = [_i64, _i64, _i64, _p, _i64, _p, _i64,
                                           _p, _i64, ctypes.c_int]
        lib.oracle_gemm_f16_nt.restype = None
        lib.oracle_gemm_f16_nt_f64.argtypes = [_i64, _i64, _i64, _p, _i64, _p, _i64,
                                               _p, _i64, ctypes.c_int]
        lib.oracle_gemm_f16_nt_f64.restype = None
        lib.oracle_gemm_f16_nt_points.argtypes = [_i64, _p, _i64, _p, _i64, _i64,
                                                  _p, _p, _p, _p]
        lib.oracle_gemm_f16_nt_points.restype = None
        lib.oracle_f64_to_f16_array.argtypes = [_i64, _p, _p]
        lib.oracle_f64_to_f16_array.restype = None
        lib.oracle_f16_to_f64_array.argtypes = [_i64, _p, _p]
        lib.oracle_f16_to_f64_array.restype = None
        lib.oracle_gemm_f16_nt_acc16.argtypes = [_i64, _i64, _i64, _p, _i64, _p, _i64,
                                                 _p, _i64, ctypes.c_int]
        lib.oracle_gemm_f16_nt_acc16.restype = None
        lib.oracle_gemm_f16_nt_acc16_points.argtypes = [_i64, _p, _i64, _p, _i64, _i64, _p, _p, _p]
        lib.oracle_gemm_f16_nt_acc16_points.restype = None
        lib.oracle_gemm_bf16_nt.argtypes = [_i64, _i64, _i64, _p, _i64, _p, _i64, _p, _i64,
                                            ctypes.c_int]
        lib.oracle_gemm_bf16_nt.restype = None
        lib.oracle_gemm_bf16_nt_points.argtypes = [_i64, _p, _i64, _p, _i64, _i64, _p, _p, _p]
        lib.oracle_gemm_bf16_nt_points.restype = None
        lib.oracle_f64_to_bf16_array.argtypes = [_i64, _p, _p]
        lib.oracle_f64_to_bf16_array.restype = None
        lib.oracle_bf16_to_f64_array.argtypes = [_i64, _p, _p]
        lib.oracle_bf16_to_f64_array.restype = None
        self.lib = lib
        self.path = lib_path

    def gemm_f16_nt(self, A: np.ndarray, B: np.ndarray, C: np.ndarray | None = None,
                    threads: int | None = None) -> np.ndarray:
        """C = RNE_fp16(A · Bᵀ) with an fp64 sequential sum per element.

        A is [M, K], B is [N, K] (row-major, any leading dimension >= K).  If C
        is given ([M, N] view, possibly of a wider buffer) it is written in place
        and nothing outside its M×N window is touched.
        """
        M, K = A.shape
        N, K2 = B.shape
        if K2 != K:
            raise ValueError("A and B disagree on K")
        if C is None:
            C = np.empty((M, N), dtype=np.float16)
        if C.shape != (M, N):
            raise ValueError("C has the wrong shape")
        pa, lda = _rows(A, "A")
        pb, ldb = _rows(B, "B")
        pc, ldc = _rows(C, "C")
        self.lib.oracle_gemm_f16_nt(M, N, K, pa, lda, pb, ldb, pc, ldc,
                                    threads or default_threads())
        return C

    def gemm_f16_nt_f64(self, A: np.ndarray, B: np.ndarray,
                        threads: int | None = None) -> np.ndarray:
        """The fp64 sums A · Bᵀ before the final rounding (same loop as above)."""
        M, K = A.shape
        N, _ = B.shape
        S = np.empty((M, N), dtype=np.float64)
        pa, lda = _rows(A, "A")
        pb, ldb = _rows(B, "B")
        self.lib.oracle_gemm_f16_nt_f64(M, N, K, pa, lda, pb, ldb, S.ctypes.data,
                                        max(N, 1), threads or default_threads())
        return S

    def gemm_f16_nt_points(self, A: np.ndarray, B: np.ndarray, rows, cols):
        """C_ref at the listed (row, col) positions, one element at a time.

        Returns (fp16 values, fp64 unrounded sums)."""
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        cols = np.ascontiguousarray(cols, dtype=np.int64)
        if rows.shape != cols.shape:
            raise ValueError("rows and cols differ in length")
        M, K = A.shape
        N, _ = B.shape
        if rows.size and (rows.min() < 0 or rows.max() >= M
                          or cols.min() < 0 or cols.max() >= N):
            raise IndexError("sample position out of range")
        out = np.empty(rows.shape, dtype=np.float16)
        out64 = np.empty(rows.shape, dtype=np.float64)
        pa, lda = _rows(A, "A")
        pb, ldb = _rows(B, "B")
        self.lib.oracle_gemm_f16_nt_points(K, pa, lda, pb, ldb, rows.size,
                                           rows.ctypes.data, cols.ctypes.data,
                                           out.ctypes.data, out64.ctypes.data)
        return out, out64

    # ---- fp16 accumulation: the accumulator rounded to fp16 every 16 k ----

    def gemm_f16_nt_acc16(self, A: np.ndarray, B: np.ndarray, C: np.ndarray | None = None,
                          threads: int | None = None) -> np.ndarray:
        """The fp16-accumulation variant: acc <- RNE_fp16(acc + the fp64 sum of
        the next 16 products), k ascending, from acc = +0; C = the last acc."""
        M, K = A.shape
        N, K2 = B.shape
        if K2 != K:
            raise ValueError("A and B disagree on K")
        if C is None:
            C = np.empty((M, N), dtype=np.float16)
        if C.shape != (M, N):
            raise ValueError("C has the wrong shape")
        pa, lda = _rows(A, "A")
        pb, ldb = _rows(B, "B")
        pc, ldc = _rows(C, "C")
        self.lib.oracle_gemm_f16_nt_acc16(M, N, K, pa, lda, pb, ldb, pc, ldc,
                                          threads or default_threads())
        return C

    def gemm_f16_nt_acc16_points(self, A: np.ndarray, B: np.ndarray, rows, cols) -> np.ndarray:
        """The fp16-accumulation variant at the listed (row, col) positions."""
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        cols = np.ascontiguousarray(cols, dtype=np.int64)
        M, K = A.shape
        N, _ = B.shape
        if rows.size and (rows.min() < 0 or rows.max() >= M
                          or cols.min() < 0 or cols.max() >= N):
            raise IndexError("sample position out of range")
        out = np.empty(rows.shape, dtype=np.float16)
        pa, lda = _rows(A, "A")
        pb, ldb = _rows(B, "B")
        self.lib.oracle_gemm_f16_nt_acc16_points(K, pa, lda, pb, ldb, rows.size, rows.ctypes.data,
                                                 cols.ctypes.data, out.ctypes.data)
        return out

    # ---- bfloat16: arrays hold bf16 bit patterns as numpy.uint16 ----------

    def gemm_bf16_nt(self, A: np.ndarray, B: np.ndarray, C: np.ndarray | None = None,
                     threads: int | None = None) -> np.ndarray:
        """C = RNE_bf16(A · Bᵀ), fp64 sequential sum per element; A [M, K] and
        B [N, K] are bf16 bit patterns (uint16), and so is the result."""
        M, K = A.shape
        N, K2 = B.shape
        if K2 != K:
            raise ValueError("A and B disagree on K")
        if C is None:
            C = np.empty((M, N), dtype=np.uint16)
        if C.shape != (M, N):
            raise ValueError("C has the wrong shape")
        pa, lda = _rows(A, "A", np.uint16)
        pb, ldb = _rows(B, "B", np.uint16)
        pc, ldc = _rows(C, "C", np.uint16)
        self.lib.oracle_gemm_bf16_nt(M, N, K, pa, lda, pb, ldb, pc, ldc,
                                     threads or default_threads())
        return C

    def gemm_bf16_nt_points(self, A: np.ndarray, B: np.ndarray, rows, cols) -> np.ndarray:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        cols = np.ascontiguousarray(cols, dtype=np.int64)
        M, K = A.shape
        N, _ = B.shape
        if rows.size and (rows.min() < 0 or rows.max() >= M
                          or cols.min() < 0 or cols.max() >= N):
            raise IndexError("sample position out of range")
        out = np.empty(rows.shape, dtype=np.uint16)
        pa, lda = _rows(A, "A", np.uint16)
        pb, ldb = _rows(B, "B", np.uint16)
        self.lib.oracle_gemm_bf16_nt_points(K, pa, lda, pb, ldb, rows.size, rows.ctypes.data,
                                            cols.ctypes.data, out.ctypes.data)
        return out

    def round_f64_to_bf16(self, x) -> np.ndarray:
        """The oracle's own fp64 -> bf16 round-to-nearest-even (uint16 bits)."""
        x = np.ascontiguousarray(x, dtype=np.float64)
        out = np.empty(x.shape, dtype=np.uint16)
        self.lib.oracle_f64_to_bf16_array(x.size, x.ctypes.data, out.ctypes.data)
        return out

    def widen_bf16_to_f64(self, h) -> np.ndarray:
        """The oracle's own bf16 -> fp64 decoding."""
        h = np.ascontiguousarray(np.asarray(h, dtype=np.uint16))
        out = np.empty(h.shape, dtype=np.float64)
        self.lib.oracle_bf16_to_f64_array(h.size, h.ctypes.data, out.ctypes.data)
        return out

    def round_f64_to_f16(self, x) -> np.ndarray:
        """The oracle's own fp64 -> fp16 round-to-nearest-even."""
        x = np.ascontiguousarray(x, dtype=np.float64)
        out = np.empty(x.shape, dtype=np.uint16)
        self.lib.oracle_f64_to_f16_array(x.size, x.ctypes.data, out.ctypes.data)
        return out.view(np.float16)

    def widen_f16_to_f64(self, h) -> np.ndarray:
        """The oracle's own fp16 -> fp64 decoding."""
        h = np.ascontiguousarray(np.asarray(h).view(np.uint16))
        out = np.empty(h.shape, dtype=np.float64)
        self.lib.oracle_f16_to_f64_array(h.size, h.ctypes.data, out.ctypes.data)
        return out


def default() -> Oracle:
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def gemm_f16_nt(A, B, C=None, threads=None):
    return default().gemm_f16_nt(A, B, C, threads)


def gemm_f16_nt_f64(A, B, threads=None):
    return default().gemm_f16_nt_f64(A, B, threads)


def gemm_f16_nt_points(A, B, rows, cols):
    return default().gemm_f16_nt_points(A, B, rows, cols)


def round_f64_to_f16(x):
    return default().round_f64_to_f16(x)


def widen_f16_to_f64(h):
    return default().widen_f16_to_f64(h)


def gemm_f16_nt_acc16(A, B, C=None, threads=None):
    return default().gemm_f16_nt_acc16(A, B, C, threads)


def gemm_f16_nt_acc16_points(A, B, rows, cols):
    return default().gemm_f16_nt_acc16_points(A, B, rows, cols)


def gemm_bf16_nt(A, B, C=None, threads=None):
    return default().gemm_bf16_nt(A, B, C, threads)


def gemm_bf16_nt_points(A, B, rows, cols):
    return default().gemm_bf16_nt_points(A, B, rows, cols)


def round_f64_to_bf16(x):
    return default().round_f64_to_bf16(x)


def widen_bf16_to_f64(h):
    return default().widen_bf16_to_f64(h)
