"""Helpers for the GPU tests: host fp16 arrays <-> device buffers with chosen pitch."""
import numpy as np


def to_device(x: np.ndarray, ld: int | None = None, fill=float("nan")):
    """Copy a [rows, cols] float16 array to cuda:0 as a [rows, cols] view of a
    [rows, ld] buffer (padding filled with `fill`).  ld defaults to cols rounded
    up to a multiple of 8 (the library's pitch rule)."""
    import torch
    rows, cols = x.shape
    if ld is None:
        ld = max(cols, 1)
        ld += (-ld) % 8
    buf = torch.full((max(rows, 1), ld), fill, dtype=torch.float16, device="cuda:0")
    if rows and cols:
        buf[:rows, :cols] = torch.from_numpy(np.ascontiguousarray(x)).to("cuda:0")
    return buf[:rows, :cols]


def to_host(t) -> np.ndarray:
    return t.detach().cpu().numpy()


def empty_out(M: int, N: int, ld: int | None = None, extra_rows: int = 0, fill=float("nan")):
    """A NaN-filled C buffer: [M + extra_rows, ld] with the [M, N] view returned
    alongside the whole buffer (for checking the untouched margins)."""
    import torch
    if ld is None:
        ld = max(N, 1)
        ld += (-ld) % 8
    buf = torch.full((M + extra_rows, ld), fill, dtype=torch.float16, device="cuda:0")
    return buf[:M, :N], buf


def lib_for(cluster_pairs: int):
    """The library that runs a cluster_pairs choice: two CTA pairs per cluster
    (A shared by TMA multicast) exist only in the single-GPU multicast build."""
    import dense_fp16_gemm_gb300 as g
    return g.library_mcast() if cluster_pairs == 2 else g.library()
