"""Build the CUDA libraries in-tree with nvcc for sm_103a (no other architecture).

Two libraries come from the same kernel source:
  libgemm_f16_nt.so        the library (no multicast copy anywhere in it);
  libgemm_f16_nt_mcast.so  the same plus clusters of two CTA pairs that share A
                           by TMA multicast, for single-GPU processes only.
The second is compiled from csrc/mcast/, which includes the first's source;
nothing in the default library's sources names a multicast load.
"""
from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_NAME = "libgemm_f16_nt.so"
LIB_PATH = os.path.join(BUILD_DIR, LIB_NAME)
MCAST_LIB_NAME = "libgemm_f16_nt_mcast.so"
MCAST_LIB_PATH = os.path.join(BUILD_DIR, MCAST_LIB_NAME)

SOURCES = [os.path.join(CSRC, "gemm_f16_nt.cu")]
DEPENDS = SOURCES + [os.path.join(CSRC, "persistent.cuh"), os.path.join(CSRC, "ptx.cuh"),
                     os.path.join(CSRC, "sched.cuh"), os.path.join(CSRC, "small_tile.cuh"),
                     os.path.join(INCLUDE, "gemm_f16_nt.h")]
MCAST_SOURCES = [os.path.join(CSRC, "mcast", "gemm_f16_nt_mcast.cu")]
MCAST_DEPENDS = DEPENDS + MCAST_SOURCES + [os.path.join(CSRC, "mcast", "tma_multicast.cuh")]

VARIANTS = {
    "default": (LIB_PATH, SOURCES, DEPENDS),
    "mcast": (MCAST_LIB_PATH, MCAST_SOURCES, MCAST_DEPENDS),
}

NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo", "-O3", "-std=c++17",
              "-Xcompiler", "-fPIC,-fvisibility=hidden", "-shared"]


def nvcc_path() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the GEMM library")


def up_to_date(variant: str = "default") -> bool:
    path, _, deps = VARIANTS[variant]
    if not os.path.exists(path):
        return False
    t = os.path.getmtime(path)
    return all(os.path.getmtime(p) <= t for p in deps)


def _command(variant: str, tmp: str, verbose: bool):
    _, sources, _ = VARIANTS[variant]
    cmd = [nvcc_path(), *NVCC_FLAGS, "-I" + INCLUDE, "-I" + CSRC, "-o", tmp, *sources]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    return cmd


def build(force: bool = False, verbose: bool = False, variants=("default",)) -> str:
    """Compile the given library variants (in parallel) if missing or older
    than their sources; returns the path of the first one."""
    variants = list(variants)
    todo = [v for v in variants if force or not up_to_date(v)]
    os.makedirs(BUILD_DIR, exist_ok=True)
    procs = []
    for v in todo:
        tmp = VARIANTS[v][0] + ".%d.tmp" % os.getpid()
        procs.append((v, tmp, subprocess.Popen(_command(v, tmp, verbose), stdout=subprocess.PIPE,
                                               stderr=subprocess.STDOUT, text=True)))
    errors = []
    for v, tmp, proc in procs:
        out, _ = proc.communicate()
        if proc.returncode != 0:
            errors.append(f"nvcc failed ({v}):\n{out}")
            continue
        if verbose:
            print(out)
        os.replace(tmp, VARIANTS[v][0])
    if errors:
        raise RuntimeError("\n".join(errors))
    return VARIANTS[variants[0]][0]


def build_all(force: bool = False, verbose: bool = False) -> None:
    """Both libraries."""
    build(force=force, verbose=verbose, variants=("default", "mcast"))


if __name__ == "__main__":
    build_all(force=True, verbose=True)
    print(LIB_PATH)
    print(MCAST_LIB_PATH)
