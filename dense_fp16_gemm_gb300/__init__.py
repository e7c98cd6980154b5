"""GB300-native dense fp16 NT GEMM:  C[M,N] = A[M,K] · B[N,K]ᵀ.

fp16 inputs, fp32 accumulation on the sm_103a tensor cores (tcgen05, TMEM),
fp16 output rounded to nearest even.  Every step runs in the CUDA library
``_build/libgemm_f16_nt.so`` (built from ``csrc/`` by ``_build_ext.build``);
this module only marshals arguments to its C ABI (declared in
``include/gemm_f16_nt.h``).  There is no CPU or other fallback: without the
library or without a compute-capability-10.3 GPU every call raises.

``library_mcast()`` loads the separately built single-GPU variant
``libgemm_f16_nt_mcast.so`` (same ABI, plus clusters of two CTA pairs that
share A by TMA multicast); pass it as ``lib=`` to the calls below.  It refuses
to load in a process that is one rank of several (WORLD_SIZE > 1).

The operation is the one the Tilus matmul-hopper tutorial computes: A is
[m_size, k_size], B is [n_size, k_size] read transposed, fp32 accumulator,
cast to fp16 ("3. Warp Specialization", §The Full Kernel).
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import _build_ext

__all__ = ["gemm_f16_nt", "gemm_bf16_nt", "gemm_f16_nt_ptr", "device_status", "device_limits", "plan", "schedule",
           "launch_plan", "device_workspace", "tile_coord", "fast_divmod", "GemmError", "Options", "Plan", "Item",
           "library", "library_mcast", "STATUS"]

STATUS = {
    0: "GEMM_OK",
    1: "GEMM_ERR_INVALID_VALUE",
    2: "GEMM_ERR_MISALIGNED",
    3: "GEMM_ERR_UNSUPPORTED_DEVICE",
    4: "GEMM_ERR_LAUNCH",
    5: "GEMM_ERR_TIMEOUT",
    6: "GEMM_ERR_SCRATCH_LIMIT",
    7: "GEMM_ERR_NOT_LOCAL",
}


class GemmError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = int(status)
        self.name = STATUS.get(self.status, "unknown")
        msg = library().gemm_f16_nt_status_string(self.status).decode()
        super().__init__(f"{what}: {msg}" if what else msg)


class Options(ctypes.Structure):
    """gemm_f16_nt_options_t (zero = default in every field)."""
    _fields_ = [("cta_group", ctypes.c_int32), ("swizzle", ctypes.c_int32),
                ("max_clusters", ctypes.c_int32), ("inject_stall", ctypes.c_int32),
                ("timeout_ns", ctypes.c_uint64), ("schedule", ctypes.c_int32),
                ("trace_items", ctypes.c_int32), ("trace", ctypes.c_void_p),
                ("cluster_pairs", ctypes.c_int32), ("a_layout", ctypes.c_int32),
                ("b_layout", ctypes.c_int32), ("accumulate", ctypes.c_int32),
                ("tile_n", ctypes.c_int32)]


class Plan(ctypes.Structure):
    """gemm_f16_nt_plan_t."""
    _fields_ = [("cta_group", ctypes.c_int32), ("tile_m", ctypes.c_int32),
                ("tile_n", ctypes.c_int32), ("block_k", ctypes.c_int32),
                ("stages", ctypes.c_int32), ("m_tiles", ctypes.c_int32),
                ("n_tiles", ctypes.c_int32), ("k_blocks", ctypes.c_int32),
                ("num_tiles", ctypes.c_int64), ("clusters", ctypes.c_int32),
                ("grid_ctas", ctypes.c_int32), ("swizzle", ctypes.c_int32),
                ("smem_bytes", ctypes.c_int32), ("tmem_cols", ctypes.c_int32),
                ("sk_tiles", ctypes.c_int32), ("cluster_pairs", ctypes.c_int32),
                ("workspace_bytes", ctypes.c_int64), ("tail_tiles", ctypes.c_int32),
                ("tail_split", ctypes.c_int32), ("split_k_off", ctypes.c_int32),
                ("split_pieces", ctypes.c_int32), ("kernel", ctypes.c_int32), ("k_order", ctypes.c_int32),
                ("claimed_tiles", ctypes.c_int32)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


class Item(ctypes.Structure):
    """gemm_f16_nt_item_t: one work item of a persistent cluster."""
    _fields_ = [("tile", ctypes.c_int32), ("m_tile", ctypes.c_int32), ("n_tile", ctypes.c_int32),
                ("kb0", ctypes.c_int32), ("kb1", ctypes.c_int32), ("kind", ctypes.c_int32),
                ("part", ctypes.c_int32), ("parts", ctypes.c_int32), ("partners", ctypes.c_int32),
                ("piece", ctypes.c_int32), ("pieces", ctypes.c_int32), ("k_down", ctypes.c_int32)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


_libs = {}
_lib_lock = threading.Lock()
_i64, _i32, _u32, _p = ctypes.c_int64, ctypes.c_int32, ctypes.c_uint32, ctypes.c_void_p


def library(path: str | None = None, variant: str = "default"):
    """Load the C-ABI library (building it first if the sources are newer).

    variant "default" is libgemm_f16_nt.so; "mcast" the single-GPU multicast
    build (see library_mcast).  Thread-safe: the first caller builds and loads
    it, the others wait."""
    key = path or variant
    lib = _libs.get(key)
    if lib is not None:
        return lib
    with _lib_lock:
        return _load_library(path, variant)


def library_mcast():
    """The single-GPU multicast build, libgemm_f16_nt_mcast.so.  Refused in a
    process that is one of several ranks; its calls also return
    GEMM_ERR_NOT_LOCAL when the process sees more than one GPU or an operand is
    not device memory of the current device."""
    if int(os.environ.get("WORLD_SIZE", "1")) > 1:
        raise RuntimeError("libgemm_f16_nt_mcast.so is for single-GPU processes (WORLD_SIZE > 1 here)")
    return library(variant="mcast")


def _load_library(path: str | None, variant: str):
    key = path or variant
    if key not in _libs:
        if path is None:
            if variant not in _build_ext.VARIANTS:
                raise ValueError(f"unknown library variant {variant!r}")
            if not _build_ext.up_to_date(variant):
                _build_ext.build(variants=(variant,))
            path = _build_ext.VARIANTS[variant][0]
        if not os.path.exists(path):
            raise RuntimeError(f"GEMM CUDA library not found at {path}")
        lib = ctypes.CDLL(path)
        sig = [_i64, _i64, _i64, _p, _i64, _p, _i64, _p, _i64, _p]
        lib.gemm_f16_nt.argtypes = sig
        lib.gemm_f16_nt.restype = ctypes.c_int
        lib.gemm_f16_nt_ex.argtypes = sig + [ctypes.POINTER(Options)]
        lib.gemm_f16_nt_ex.restype = ctypes.c_int
        lib.gemm_f16_nt_noalloc.argtypes = sig
        lib.gemm_f16_nt_noalloc.restype = ctypes.c_int
        lib.gemm_bf16_nt.argtypes = sig
        lib.gemm_bf16_nt.restype = ctypes.c_int
        lib.gemm_bf16_nt_ex.argtypes = sig + [ctypes.POINTER(Options)]
        lib.gemm_bf16_nt_ex.restype = ctypes.c_int
        lib.gemm_f16_nt_device_status.argtypes = [_p, ctypes.POINTER(_u32)]
        lib.gemm_f16_nt_device_status.restype = ctypes.c_int
        lib.gemm_f16_nt_debug_status.argtypes = [_p]
        lib.gemm_f16_nt_debug_status.restype = ctypes.c_int
        lib.gemm_f16_nt_device_workspace.argtypes = [ctypes.POINTER(_i32), ctypes.POINTER(_i64)]
        lib.gemm_f16_nt_device_workspace.restype = ctypes.c_int
        lib.gemm_f16_nt_multicast_available.argtypes = []
        lib.gemm_f16_nt_multicast_available.restype = ctypes.c_int32
        lib.gemm_f16_nt_status_string.argtypes = [ctypes.c_int]
        lib.gemm_f16_nt_status_string.restype = ctypes.c_char_p
        lib.gemm_f16_nt_plan.argtypes = [_i64, _i64, _i64, _i32, _i32, ctypes.POINTER(Options),
                                         ctypes.POINTER(Plan)]
        lib.gemm_f16_nt_plan.restype = ctypes.c_int
        lib.gemm_f16_nt_launch_plan.argtypes = [_i64, _i64, _i64, _i64, _i64, _p, ctypes.POINTER(Options),
                                                ctypes.POINTER(Plan)]
        lib.gemm_f16_nt_launch_plan.restype = ctypes.c_int
        lib.gemm_f16_nt_schedule.argtypes = [_i64, _i64, _i64, _i32, _i32, ctypes.POINTER(Options), _i32,
                                             ctypes.POINTER(Item), _i32, ctypes.POINTER(_i32)]
        lib.gemm_f16_nt_schedule.restype = ctypes.c_int
        lib.gemm_f16_nt_tile_coord.argtypes = [_i64, _i32, _i32, _i32, ctypes.POINTER(_i32),
                                               ctypes.POINTER(_i32)]
        lib.gemm_f16_nt_tile_coord.restype = ctypes.c_int
        lib.gemm_f16_nt_fast_divmod.argtypes = [_u32, _u32, ctypes.POINTER(_u32),
                                                ctypes.POINTER(_u32)]
        lib.gemm_f16_nt_fast_divmod.restype = ctypes.c_int
        lib.gemm_f16_nt_device_limits.argtypes = [ctypes.POINTER(_i32)] * 4
        lib.gemm_f16_nt_device_limits.restype = ctypes.c_int
        _libs[key] = lib
    return _libs[key]


def _check(status: int, what: str):
    if status != 0:
        raise GemmError(status, what)


def gemm_f16_nt_ptr(M: int, N: int, K: int, a_ptr: int, lda: int, b_ptr: int, ldb: int,
                    c_ptr: int, ldc: int, stream: int = 0, options: Options | None = None,
                    bf16: bool = False, lib=None) -> None:
    """Raw call: device pointers (ints), leading dimensions in elements, a
    cudaStream_t handle (int); bf16=True calls the bfloat16 entry points; `lib`
    a loaded library (default: library()).  Raises GemmError on a non-OK
    status."""
    lib = lib or library()
    name = "gemm_bf16_nt" if bf16 else "gemm_f16_nt"
    if options is None:
        st = getattr(lib, name)(M, N, K, a_ptr, lda, b_ptr, ldb, c_ptr, ldc, stream)
    else:
        st = getattr(lib, name + "_ex")(M, N, K, a_ptr, lda, b_ptr, ldb, c_ptr, ldc, stream,
                                        ctypes.byref(options))
    _check(st, name)


def _rows(t, name, dtype=None):
    import torch
    dtype = dtype or torch.float16
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype or t.dim() != 2:
        raise TypeError(f"{name} must be a 2-D {dtype} tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device")
    if t.shape[1] > 1 and t.stride(1) != 1:
        raise ValueError(f"{name} must have unit stride along its last dimension")
    if t.shape[0] > 1:
        ld = t.stride(0)
    else:  # a single row: the pitch is never used to address memory
        ld = max(t.shape[1], 1)
        ld += (-ld) % 8
    return t.data_ptr(), ld


def _call(A, B, C, stream, options, a_layout, b_layout, bf16, lib=None):
    import torch
    dt = torch.bfloat16 if bf16 else torch.float16
    M, K = (A.shape[1], A.shape[0]) if a_layout else tuple(A.shape)
    N, K2 = (B.shape[1], B.shape[0]) if b_layout else tuple(B.shape)
    if K2 != K:
        raise ValueError(f"A and B disagree on K ({K} vs {K2})")
    if C is None:   # row pitch rounded up to 8 elements (16 bytes), as the kernel needs
        C = torch.empty((M, N + (-N) % 8), dtype=dt, device=A.device)[:, :N]
    if tuple(C.shape) != (M, N):
        raise ValueError(f"C must be [{M}, {N}]")
    if stream is None:
        stream = torch.cuda.current_stream(A.device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    if a_layout or b_layout:
        options = options if options is not None else Options()
        options.a_layout, options.b_layout = a_layout, b_layout
    pa, lda = _rows(A, "A", dt)
    pb, ldb = _rows(B, "B", dt)
    pc, ldc = _rows(C, "C", dt)
    with torch.cuda.device(A.device):
        gemm_f16_nt_ptr(M, N, K, pa, lda, pb, ldb, pc, ldc, handle, options, bf16=bf16, lib=lib)
    return C


def gemm_f16_nt(A, B, C=None, *, stream=None, options: Options | None = None,
                a_layout: int = 0, b_layout: int = 0, lib=None):
    """C[m, n] = sum_k A(m, k) B(n, k) for CUDA float16 tensors.

    A is [M, K] (a_layout 0) or [K, M] (a_layout 1); B is [N, K] (b_layout 0)
    or [K, N] (b_layout 1) — with b_layout 1 this is C = A @ B.  C, if given,
    is an [M, N] float16 view (its row stride may exceed N) and is
    overwritten; otherwise a new [M, N] view of a buffer whose row pitch is N
    rounded up to a multiple of 8 is returned.  The call is
    asynchronous on `stream` (default: torch's current stream).  `lib`: a
    loaded library (default: library(); library_mcast() for the multicast
    build)."""
    return _call(A, B, C, stream, options, a_layout, b_layout, False, lib)


def gemm_bf16_nt(A, B, C=None, *, stream=None, options: Options | None = None,
                 a_layout: int = 0, b_layout: int = 0, lib=None):
    """As gemm_f16_nt for CUDA bfloat16 tensors (fp32 accumulation, bf16 result)."""
    return _call(A, B, C, stream, options, a_layout, b_layout, True, lib)


def device_status(stream=None, lib=None) -> int:
    """Synchronise `stream`, then read and clear the device watchdog word.
    Returns the word (0 = no wait expired); raises GemmError on CUDA errors."""
    handle = 0
    if stream is not None:
        handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    flags = _u32(0)
    st = (lib or library()).gemm_f16_nt_device_status(handle, ctypes.byref(flags))
    if st not in (0, 5):
        raise GemmError(st, "gemm_f16_nt_device_status")
    return int(flags.value)


def device_limits(lib=None) -> dict:
    """SM count and resident CTA pairs / CTAs of the current device."""
    a, b, c, d = _i32(0), _i32(0), _i32(0), _i32(0)
    _check((lib or library()).gemm_f16_nt_device_limits(ctypes.byref(a), ctypes.byref(b), ctypes.byref(c),
                                                        ctypes.byref(d)), "gemm_f16_nt_device_limits")
    return {"sms": a.value, "resident_pairs": b.value, "resident_ctas": c.value,
            "resident_pair_pairs": d.value}


def plan(M: int, N: int, K: int, num_sms: int = 152, max_clusters: int = 0,
         options: Options | None = None, lib=None) -> dict:
    """The launch plan for a problem (host computation only, no GPU needed)."""
    out = Plan()
    st = (lib or library()).gemm_f16_nt_plan(M, N, K, num_sms, max_clusters,
                                             ctypes.byref(options) if options is not None else None,
                                             ctypes.byref(out))
    _check(st, "gemm_f16_nt_plan")
    return out.as_dict()


def launch_plan(M: int, N: int, K: int, lda: int | None = None, ldb: int | None = None, stream=None,
                options: Options | None = None, lib=None) -> dict:
    """The plan a call would launch right now on the current device and
    `stream` (default: the legacy default stream): resident clusters, the
    automatic choices for lda/ldb (default K), and split_k_off (1: the stream
    is capturing, 2: no stream-K workspace reserved)."""
    handle = 0
    if stream is not None:
        handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    out = Plan()
    st = (lib or library()).gemm_f16_nt_launch_plan(
        M, N, K, K if lda is None else lda, K if ldb is None else ldb, handle,
        ctypes.byref(options) if options is not None else None, ctypes.byref(out))
    _check(st, "gemm_f16_nt_launch_plan")
    return out.as_dict()


def device_workspace(lib=None) -> dict:
    """Stream-K workspace slots reserved on the current device, and their size."""
    n, b = _i32(0), _i64(0)
    _check((lib or library()).gemm_f16_nt_device_workspace(ctypes.byref(n), ctypes.byref(b)),
           "gemm_f16_nt_device_workspace")
    return {"slots": n.value, "bytes_per_slot": b.value}


def schedule(M: int, N: int, K: int, cluster: int, num_sms: int = 152, max_clusters: int = 0,
             options: Options | None = None, lib=None) -> list:
    """The work items persistent cluster `cluster` runs, in order, as dicts
    (host computation with the kernel's own schedule code; no GPU needed)."""
    lib = lib or library()
    opt = ctypes.byref(options) if options is not None else None
    n = _i32(0)
    _check(lib.gemm_f16_nt_schedule(M, N, K, num_sms, max_clusters, opt, cluster, None, 0, ctypes.byref(n)),
           "gemm_f16_nt_schedule")
    items = (Item * max(1, n.value))()
    _check(lib.gemm_f16_nt_schedule(M, N, K, num_sms, max_clusters, opt, cluster, items, n.value,
                                    ctypes.byref(n)), "gemm_f16_nt_schedule")
    return [items[i].as_dict() for i in range(n.value)]


def tile_coord(linear: int, m_tiles: int, n_tiles: int, swizzle: int):
    m, n = _i32(0), _i32(0)
    st = library().gemm_f16_nt_tile_coord(linear, m_tiles, n_tiles, swizzle, ctypes.byref(m),
                                          ctypes.byref(n))
    _check(st, "gemm_f16_nt_tile_coord")
    return m.value, n.value


def fast_divmod(n: int, d: int):
    q, r = _u32(0), _u32(0)
    st = library().gemm_f16_nt_fast_divmod(n, d, ctypes.byref(q), ctypes.byref(r))
    _check(st, "gemm_f16_nt_fast_divmod")
    return q.value, r.value
