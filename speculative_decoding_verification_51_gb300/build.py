"""Compile the CUDA library in-tree for sm_103a with nvcc.

Each translation unit under ``csrc/`` is compiled in parallel, then linked
into ``_build/libspecverify_<machine>.so`` (CUDA runtime linked statically).
The library is rebuilt when any source or header is newer than it.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import platform
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
SOURCES = ["plan.cu", "row_stats.cu", "sample.cu", "verify.cu", "tree.cu", "lmhead.cu", "host_io.cu",
           "api.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", f"-I{INCLUDE}"]


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if c and (os.path.sep not in c or os.path.exists(c)):
            return c
    return "nvcc"


def lib_path() -> str:
    return os.path.join(BUILD, f"libspecverify_{platform.machine()}.so")


def _inputs() -> list[str]:
    return (glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh"))
            + glob.glob(os.path.join(INCLUDE, "*.h")))


def extra_flags() -> list[str]:
    """Extra nvcc flags from SPEC_VERIFY_NVCC_EXTRA (e.g. launch-shape -D overrides)."""
    return os.environ.get("SPEC_VERIFY_NVCC_EXTRA", "").split()


def _stamp() -> str:
    return lib_path() + ".flags"


def up_to_date() -> bool:
    out = lib_path()
    if not os.path.exists(out) or not os.path.exists(_stamp()):
        return False
    if open(_stamp()).read() != " ".join(extra_flags()):
        return False
    return os.path.getmtime(out) >= max(os.path.getmtime(p) for p in _inputs())


def build(force: bool = False, ptxas_verbose: bool = False) -> str:
    """Build the library if needed; return its path."""
    out = lib_path()
    if not force and up_to_date():
        return out
    objdir = os.path.join(BUILD, f"obj_{platform.machine()}")
    os.makedirs(objdir, exist_ok=True)
    extra = (["-Xptxas", "-v"] if ptxas_verbose else []) + extra_flags()

    def compile_one(src: str) -> tuple[str, str]:
        obj = os.path.join(objdir, src.replace(".cu", ".o"))
        cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    tmp = f"{out}.{os.getpid()}.tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *[o for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, out)
    with open(_stamp(), "w") as f:
        f.write(" ".join(extra_flags()))
    if ptxas_verbose:
        for (_, log), src in zip(results, SOURCES):
            print(f"== {src}\n{log}")
    return out


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, ptxas_verbose="-v" in sys.argv))
