"""Seeded synthetic inputs for the fp16 NT GEMM workloads.

This module draws numbers and nothing else: it holds no part of the
multiply.  Both the CUDA path's tests and benchmark and the CPU oracle read the
arrays it makes, so the two sides always see the same fp16 bit patterns.

Recipe: values are drawn in float32 from numpy's PCG64 generator seeded per
operand (uniform: a float32 in [0, 1) scaled to [lo, hi); normal: standard
normal float32 times sigma plus mean; integers: uniform on {lo..hi}), then
rounded to float16 with numpy's round-to-nearest-even cast.

The workloads follow the shapes the tutorial measures (Tilus matmul-hopper
tutorial, "6. Register Reallocation, Multicast, and a Persistent Kernel",
§Performance: M = N = K = 8192, fp16 in and out, fp32 accumulation) plus four
more: a small case, 4096³, a ragged shape with no dimension a multiple of
64/128/256 (once with uniform floats and once with small integers, where the
product is exact), and an LLM MLP up-projection shape with Gaussian operands.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    dist_a: tuple      # ("uniform", lo, hi) | ("normal", mean, std) | ("int", lo, hi)
    dist_b: tuple
    seed_a: int
    seed_b: int

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def compulsory_bytes(self) -> int:
        return 2 * (self.M * self.K + self.N * self.K + self.M * self.N)


U = ("uniform", -1.0, 1.0)
I2 = ("int", -2, 2)

WORKLOADS = {
    "gemm_256": Workload("gemm_256", 256, 256, 256, U, U, 1, 2),
    "gemm_4096": Workload("gemm_4096", 4096, 4096, 4096, U, U, 3, 4),
    "gemm_8192": Workload("gemm_8192", 8192, 8192, 8192, U, U, 5, 6),
    "ragged_4000x3000x5000": Workload("ragged_4000x3000x5000", 4000, 3000, 5000, U, U, 7, 8),
    "ragged_int_4000x3000x5000": Workload("ragged_int_4000x3000x5000", 4000, 3000, 5000,
                                          I2, I2, 9, 10),
    "mlp_up_16384x14336x4096": Workload("mlp_up_16384x14336x4096", 16384, 14336, 4096,
                                        ("normal", 0.0, 1.0), ("normal", 0.0, 0.02), 11, 12),
    # small, latency-bound shapes beside the configs: square, short-and-wide,
    # and few tiles with deep k
    "gemm_1024": Workload("gemm_1024", 1024, 1024, 1024, U, U, 13, 14),
    "gemm_512x4096x4096": Workload("gemm_512x4096x4096", 512, 4096, 4096, U, U, 15, 16),
    "gemm_256x256x4096": Workload("gemm_256x256x4096", 256, 256, 4096, U, U, 17, 18),
}


def draw(shape, dist: tuple, seed: int, ld: int | None = None) -> np.ndarray:
    """A float16 array of `shape` (rows, cols) drawn from `dist` with `seed`.

    If `ld` > cols, the array is a [rows, cols] view of a [rows, ld] buffer whose
    padding columns hold a fixed non-finite marker (fp16 0x7e00, a NaN), so that
    any read of the padding shows up in a result.
    """
    rows, cols = shape
    rng = np.random.Generator(np.random.PCG64(seed))
    kind = dist[0]
    if kind == "uniform":
        x = rng.random(size=(rows, cols), dtype=np.float32)      # [0, 1)
        x *= np.float32(dist[2] - dist[1])
        x += np.float32(dist[1])
    elif kind == "normal":
        x = rng.standard_normal(size=(rows, cols), dtype=np.float32)
        x = (x * np.float32(dist[2]) + np.float32(dist[1])).astype(np.float32)
    elif kind == "int":
        x = rng.integers(dist[1], dist[2] + 1, size=(rows, cols), dtype=np.int8).astype(np.float32)
    else:
        raise ValueError(f"unknown distribution {kind!r}")
    h = x.astype(np.float16)
    if ld is None or ld == cols:
        return h
    if ld < cols:
        raise ValueError("ld < cols")
    buf = np.full((rows, ld), np.float16(np.nan), dtype=np.float16)
    buf[:, :cols] = h
    return buf[:, :cols]


def draw_bf16(shape, dist: tuple, seed: int, ld: int | None = None) -> np.ndarray:
    """Like `draw`, but rounded to bfloat16: the result holds bf16 bit
    patterns as uint16 (numpy has no bfloat16 type).  The float32 values are
    rounded to nearest, ties to even, on their bit pattern; padding columns
    (ld > cols) hold a bf16 NaN (0x7fc0)."""
    rows, cols = shape
    rng = np.random.Generator(np.random.PCG64(seed))
    kind = dist[0]
    if kind == "uniform":
        x = rng.random(size=(rows, cols), dtype=np.float32)
        x *= np.float32(dist[2] - dist[1])
        x += np.float32(dist[1])
    elif kind == "normal":
        x = rng.standard_normal(size=(rows, cols), dtype=np.float32)
        x = (x * np.float32(dist[2]) + np.float32(dist[1])).astype(np.float32)
    elif kind == "int":
        x = rng.integers(dist[1], dist[2] + 1, size=(rows, cols), dtype=np.int8).astype(np.float32)
    else:
        raise ValueError(f"unknown distribution {kind!r}")
    u = x.view(np.uint32).astype(np.uint64)
    h = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)   # finite inputs only
    if ld is None or ld == cols:
        return h
    if ld < cols:
        raise ValueError("ld < cols")
    buf = np.full((rows, ld), 0x7FC0, dtype=np.uint16)
    buf[:, :cols] = h
    return buf[:, :cols]


def operands(w: Workload):
    """(A [M,K], B [N,K]) for a workload, contiguous float16."""
    return draw((w.M, w.K), w.dist_a, w.seed_a), draw((w.N, w.K), w.dist_b, w.seed_b)


def draw_device_ints(shape, lo: int, hi: int, seed: int, device):
    """A float16 torch tensor of `shape` on `device`, integers uniform on
    {lo..hi} from torch's own generator for that device seeded with `seed`.

    For operands too large to draw on the host (tens of GB); reproducible for a
    given seed, device type and torch version.  Rows can be copied to the host
    for the oracle."""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    return torch.randint(lo, hi + 1, tuple(shape), generator=gen, device=device, dtype=torch.float16)
